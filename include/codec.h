/*
 * codec.h - C ABI of the GB300 (sm_103a) streaming codec-to-waveform decoder.
 *
 * The decoder turns residual-VQ code frames (12.5 Hz, Q codebooks) into 24 kHz
 * audio, 1920 samples per frame, through: codebook embedding sum -> causal
 * Conv1d -> sliding-window causal transformer -> 2x2 latent upsampling ->
 * BigVGAN stages (Snake -> transposed conv -> multi-receptive-field residual
 * blocks) -> Snake -> conv -> tanh (vllm-omni "Edge TTS design", section 1.3).
 * It decodes chunk by chunk and carries each stream's state between calls:
 * every causal conv's left context and the attention window's keys/values
 * (section 1.3 "Cross-chunk state"; blixt/phonon "Speed" item 7), so decoding
 * a stream in chunks of any sizes gives the same audio as one full decode.
 *
 * Conventions
 *   - Every entry point returns a codec_status; nothing aborts the process.
 *   - Pointers documented "device" are CUDA device pointers on the device that
 *     was current at codec_create; "host" pointers are ordinary host memory.
 *   - stream arguments are cudaStream_t values passed as void*; NULL means the
 *     legacy default stream.
 *   - Argument checks happen before anything is enqueued: a call that returns
 *     an error status other than CODEC_ERR_CUDA has enqueued no GPU work.
 *   - codec_t is immutable after creation and may be shared by threads.  A
 *     codec_state_t must be used by one host thread at a time.
 *   - All device memory is allocated in codec_create / codec_state_create
 *     (blixt/phonon "Speed" item 4: nothing is allocated per request).
 */
#ifndef GB300_CODEC_H
#define GB300_CODEC_H

#include <stdint.h>

#if defined(__GNUC__)
#define CODEC_API __attribute__((visibility("default")))
#else
#define CODEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum codec_status {
    CODEC_OK = 0,
    CODEC_ERR_NULL = 1,        /* a required pointer argument is NULL */
    CODEC_ERR_CONFIG = 2,      /* configuration invalid or unsupported */
    CODEC_ERR_WEIGHTS = 3,     /* weight blob length does not match the config */
    CODEC_ERR_ARG = 4,         /* an argument is out of range, or stream ids repeat */
    CODEC_ERR_CAPACITY = 5,    /* request exceeds max_streams, max_chunk_frames or max_batch_frames */
    CODEC_ERR_OOM = 6,         /* a device allocation failed (create calls only) */
    CODEC_ERR_CUDA = 7,        /* a CUDA runtime/driver call failed */
    CODEC_ERR_NO_DEVICE = 8    /* no usable sm_103 device */
} codec_status;

/* Sticky per-stream device error bits, read with codec_state_query. */
#define CODEC_STREAM_ERR_BAD_CODE 1u   /* a code outside [0, V): that frame's embedding was zeroed */
/* State-wide: a tensor-core kernel gave up on one of its bounded waits in a
 * call since the last reset of all slots; the audio of that call is not
 * valid.  Reported on every slot's query; cleared by codec_state_reset with
 * stream_ids == NULL. */
#define CODEC_STREAM_ERR_KERNEL_TIMEOUT 0x80000000u

typedef enum codec_precision {
    /* fp32 operands on CUDA cores for every stage. */
    CODEC_PRECISION_FP32 = 0,
    /* Dense contractions (conv, transposed conv, linear with >= 64 channels) on
     * tcgen05 tensor cores with both operands split into fp16 hi + lo parts and
     * three MMAs (hi*hi + hi*lo + lo*hi) accumulated in fp32 in TMEM; the rest
     * on CUDA cores in fp32. */
    CODEC_PRECISION_FP16X3 = 1,
    /* The same contractions in a single fp16 pass (hi*hi only: both operands
     * rounded to fp16, fp32 accumulation).  Faster, but approximate: on the
     * random-weight decoders it misses the 1e-3 waveform bound of the other
     * two modes (its error against the fp64 reference is reported, not
     * bounded).  The reduced-precision decoder mode of the vllm-omni "Edge TTS
     * design" page, section 1.5 (quality row: no lower than fp16 for the
     * decoder). */
    CODEC_PRECISION_FP16 = 2
} codec_precision;

/*
 * Decoder shape and capacity.  The layer list is fixed by the stage order
 * above; these fields size it.
 */
typedef struct codec_config {
    int32_t Q, V, E;          /* codebooks, entries per codebook, codebook width */
    int32_t pre_k;            /* kernel of the causal Conv1d E -> d */
    int32_t d, heads, ffn;    /* transformer width, heads (d % heads == 0), MLP width */
    int32_t layers, window;   /* transformer layers; keys per query (itself included), 1..256 */
    int32_t n_up, up_k, up_s; /* latent transposed convs: count (1..4), kernel, stride; up_k == 2*up_s */
    int32_t up_ch[4];         /* their output channels; up_ch[n_up-1] = C_0 */
    int32_t n_stages;         /* BigVGAN stages (1..8) */
    int32_t strides[8];       /* stage strides s_i; the stage's ConvT kernel is 2*s_i */
    int32_t ch[8];            /* stage output channels C_1..C_n */
    int32_t n_rb;             /* resblocks per stage (1..3), averaged when > 1 */
    int32_t rb_k[4];          /* their kernels (odd) */
    int32_t n_dil;            /* dilations per resblock (1..4) */
    int32_t dil[4];
    int32_t final_k;          /* kernel of the final conv C_n -> 1 */
    float rms_eps;
    int32_t max_streams;      /* default stream slots for codec_state_create(n_streams = 0) */
    int32_t max_chunk_frames; /* largest n_frames[b] accepted in one call (>= 1) */
    int32_t max_batch_frames; /* largest sum of n_frames over one call (>= max_chunk_frames) */
    int32_t precision;        /* codec_precision */
    /* Latent-input variant (blixt/phonon "Weights", "Speed" item 7): 0 for RVQ
     * code input (Q, V, E, pre_k as above).  L > 0 (a multiple of 4): frames
     * of L continuous latent channels come in (codec_decode_latents), are
     * denormalised, projected 1x1 to d and upsampled tf_up times by a causal
     * depthwise transposed conv (kernel 2 tf_up); the transformer then runs
     * at tf_up rows per frame (window and positions count those rows), and
     * n_up may be 0 (C_0 = d).  Q, V, E, pre_k are ignored. */
    int32_t latent_dim;
    int32_t tf_up;            /* latent input: 1..64 */
} codec_config;

typedef struct codec_stream_info {
    int64_t frames_decoded;   /* frames decoded since the last reset */
    uint32_t error_bits;      /* sticky CODEC_STREAM_ERR_* bits since the last reset */
    int32_t reserved;
} codec_stream_info;

typedef struct codec_s codec_t;
typedef struct codec_state_s codec_state_t;

/* Number of fp32 values of the weight blob for cfg (-1 if cfg is invalid).
 * Blob order and layouts (PyTorch layouts, fp32):
 *   Q codebooks [V][E]; pre-conv weight [d][E][pre_k], bias [d];
 *   per layer: attention RMSNorm gain [d], Wq, Wk, Wv, Wo [d][d] ([out][in]),
 *     MLP RMSNorm gain [d], W1 [ffn][d], W2 [d][ffn];
 *   final RMSNorm gain [d];
 *   per latent ConvT: weight [Cin][Cout][up_k], bias [Cout];
 *   per stage: Snake alpha [Cin], ConvT weight [Cin][Cout][2 s], bias [Cout],
 *     then per resblock j, per dilation i: Snake alpha [C], conv weight
 *     [C][C][rb_k[j]], bias [C];
 *   final Snake alpha [C_n], conv weight [1][C_n][final_k], bias [1].
 * Latent input: in place of the codebooks and the pre-conv, mu [L], sigma
 *   [L] (z = x sigma + mu), projection [d][L] (1x1, no bias), depthwise
 *   transposed-conv taps [d][1][2 tf_up], bias [d]. */
CODEC_API int64_t codec_weight_floats(const codec_config* cfg);

/* Validate cfg, repack the weights for the kernels and upload them to the
 * current CUDA device.  weights: host, codec_weight_floats(cfg) floats; the
 * library copies them, and the caller may free them on return.
 * Errors: CODEC_ERR_NULL, CODEC_ERR_CONFIG, CODEC_ERR_WEIGHTS,
 * CODEC_ERR_NO_DEVICE, CODEC_ERR_OOM, CODEC_ERR_CUDA.  On error *out is NULL. */
CODEC_API codec_status codec_create(const codec_config* cfg, const float* weights, int64_t n_floats,
                          codec_t** out);

/*
 * The weight blob in the blixt/phonon "Weights" storage format: every tensor
 * of 16,384 values or more as int8 with one f16 scale per 32 values along the
 * rows of its converted layout (scale = max |value| / 127 of the f16-rounded
 * values, round half to even), every other tensor as f16.  Layout, tensor by
 * tensor in blob order, each part starting on a 4-byte boundary:
 *   quantised: int8 q [R][L], then f16 scale [R][ceil(L / 32)], value (r, c) =
 *              q[r][c] * scale[r][c / 32];
 *   other:     f16 values in the blob's own layout.
 * Converted rows: codebooks and linears [out][in]; convolutions [out][tap][in];
 * transposed convolutions [out][phase][tap][in] with kernel index phase +
 * tap * stride.  About a quarter of the fp32 blob's size.
 * codec_q8_bytes: the file's size for cfg (-1 if cfg is invalid).
 * codec_create_q8: as codec_create, from such a file (host memory, copied):
 * a kernel expands it on the device to the fp32 blob (int8 x f16 is exact in
 * fp32), from which the codec is built; the decode then runs on exactly the
 * dequantised weights, in cfg.precision.  Errors as codec_create
 * (CODEC_ERR_WEIGHTS for a wrong size).
 */
CODEC_API int64_t codec_q8_bytes(const codec_config* cfg);
CODEC_API codec_status codec_create_q8(const codec_config* cfg, const void* q8, int64_t n_bytes, codec_t** out);

/* Free the weights.  All states created from it must be destroyed first and
 * their GPU work finished. */
CODEC_API void codec_destroy(codec_t* codec);

/* Samples per frame (the product of all upsampling strides; 1920 for the
 * 12.5 Hz -> 24 kHz decoder). */
CODEC_API int32_t codec_samples_per_frame(const codec_t* codec);

/* Allocate n_streams stream slots (0 = cfg.max_streams) plus the per-call
 * workspace, all reset.  Errors: CODEC_ERR_NULL, CODEC_ERR_ARG, CODEC_ERR_OOM,
 * CODEC_ERR_CUDA. */
CODEC_API codec_status codec_state_create(codec_t* codec, int32_t n_streams, codec_state_t** out);

/* Free a state.  Synchronises with its device work first. */
CODEC_API void codec_state_destroy(codec_state_t* state);

/* Reset streams: clear their carried context, frame counters and error bits.
 * This is the abort / start-of-utterance operation (vllm-omni "Edge TTS
 * design", section 2.2: IDecoderAdapter::reset; section 2.2 step 4: abort).
 * stream_ids: host [n] slot ids, or NULL for every slot (n ignored).  Enqueued
 * on stream; ordered with decode calls on the same stream.
 * Errors: CODEC_ERR_NULL, CODEC_ERR_ARG, CODEC_ERR_CUDA. */
CODEC_API codec_status codec_state_reset(codec_state_t* state, const int32_t* stream_ids, int32_t n,
                               void* stream);

/*
 * Decode one chunk for each of B streams in one launch sequence.
 *   codes      device int32 [B][Q][T_max]; stream b's frames are columns 0..n_frames[b]-1.
 *   n_frames   host int32 [B], each in [0, min(T_max, max_chunk_frames)];
 *              sum <= max_batch_frames.  0 leaves the stream untouched.
 *   stream_ids host int32 [B] distinct slot ids, or NULL for slots 0..B-1.
 *   audio      device float [B][T_max * samples_per_frame]; samples
 *              0..n_frames[b]*spf-1 of row b are written, the rest untouched.
 * Each stream continues from its carried state, so its audio is final when
 * written and chunk sizes may change from call to call (vllm-omni "Edge TTS
 * design", section 1.4: 1 frame, then 25-frame chunks with the 72-frame
 * window carried).  The call returns once the work is enqueued on stream; the
 * caller keeps codes and audio alive until that work completes.
 * Errors (nothing enqueued): CODEC_ERR_NULL, CODEC_ERR_ARG (B < 1, T_max < 1,
 * n_frames out of range, slot id out of range or repeated),
 * CODEC_ERR_CAPACITY, CODEC_ERR_CONFIG (a latent-input codec);
 * CODEC_ERR_CUDA if a launch fails.
 * Codes outside [0, V) do not fail the call: they set the stream's sticky
 * CODEC_STREAM_ERR_BAD_CODE bit and that frame's embedding is zero.
 */
CODEC_API codec_status codec_decode_chunk(codec_state_t* state, const int32_t* codes, const int32_t* n_frames,
                                const int32_t* stream_ids, int32_t B, int32_t T_max, float* audio,
                                void* stream);

/* codec_decode_chunk for the latent-input variant (cfg.latent_dim = L > 0;
 * else CODEC_ERR_CONFIG): latents device float [B][T_max][L], stream b's
 * frames are rows 0 .. n_frames[b] - 1 of batch entry b.  The front end
 * (denormalise, 1x1 projection folded into the depthwise upsampling's phase
 * GEMM) replaces the codebook sum and the pre-conv; everything else,
 * arguments, errors and the carried state included, is as codec_decode_chunk.
 * pre_tanh as in codec_decode_chunk_ex (may be NULL).  Chunks of any sizes
 * share one state (blixt/phonon "Speed" item 7: chunks of 1, 2, 4, 8 frames). */
CODEC_API codec_status codec_decode_latents(codec_state_t* state, const float* latents, const int32_t* n_frames,
                                            const int32_t* stream_ids, int32_t B, int32_t T_max, float* audio,
                                            float* pre_tanh, void* stream);

/* As codec_decode_chunk, and also writes the final conv's output before tanh
 * to pre_tanh (device float, same layout as audio; may be NULL).  For
 * verification: the tanh saturates most samples of a random-weight decoder. */
CODEC_API codec_status codec_decode_chunk_ex(codec_state_t* state, const int32_t* codes,
                                   const int32_t* n_frames, const int32_t* stream_ids, int32_t B,
                                   int32_t T_max, float* audio, float* pre_tanh, void* stream);

/* The codebook embedding sum alone (the first stage of codec_decode_chunk),
 * for verification: emb is device float [sum(n_frames)][E], the frames of the
 * batch rows with n_frames[b] > 0 packed in batch order.  Arguments and
 * checks as codec_decode_chunk; no carried context changes, but a code
 * outside [0, V) sets the stream's sticky bad-code bit as in a decode. */
CODEC_API codec_status codec_embed_chunk(codec_state_t* state, const int32_t* codes, const int32_t* n_frames,
                               const int32_t* stream_ids, int32_t B, int32_t T_max, float* emb,
                               void* stream);

/*
 * Recompute-mode decode: the server schedule of the vllm-omni "Edge TTS
 * design" page, section 1.4 (each chunk after the first is decoded "with
 * 72-frame left ctx"), where a call re-decodes its left context from an empty
 * state and keeps only the new frames' audio.  For each batch entry b with
 * n_new[b] > 0, its slot is reset, frames 0 .. n_ctx[b] + n_new[b] - 1 of row b
 * of codes are decoded from the empty state, and only the audio of the last
 * n_new[b] frames is written, to samples 0 .. n_new[b] * spf - 1 of row b of
 * audio (and of pre_tanh, device float of audio's layout, or NULL).  The
 * context frames' audio is computed and dropped.  Afterwards the slot carries
 * the state after all n_ctx[b] + n_new[b] frames, so a carried-mode
 * codec_decode_chunk may follow.  Entries with n_new[b] == 0 are left alone.
 * With the decoder's exact causality, the kept audio equals the last n_new[b]
 * frames of a full decode of those n_ctx[b] + n_new[b] frames from reset.
 *   codes   device int32 [B][Q][T_max]; n_ctx, n_new: host int32 [B], each
 *           >= 0 with n_ctx[b] + n_new[b] <= min(T_max, max_chunk_frames);
 *           the sum over entries with n_new[b] > 0 <= max_batch_frames.
 * Errors as codec_decode_chunk (nothing enqueued, not even the reset). */
CODEC_API codec_status codec_decode_recompute(codec_state_t* state, const int32_t* codes, const int32_t* n_ctx,
                                              const int32_t* n_new, const int32_t* stream_ids, int32_t B,
                                              int32_t T_max, float* audio, float* pre_tanh, void* stream);

/*
 * Chunk schedules of the streaming orchestrator (vllm-omni "Edge TTS design",
 * section 2.2 "Orchestrator loop": the measured default of 1 frame then 25,
 * the codec_chunk_ramp example 4, 4, 8, 16, 25, and codec_chunk_adaptive).
 * codec_chunk_frames returns the frames of chunk `index` (0 = the first),
 * given the frames already delivered before it, or 0 for an invalid schedule.
 *   FIXED     chunk 0: first; later chunks: steady.
 *   RAMP      chunk i < n_ramp: ramp[i]; later chunks: steady.
 *   ADAPTIVE  chunk 0: min(first, steady); chunk i >= 1: the audio already
 *             delivered, in frames, capped at steady (at least 1).  From a
 *             producer that makes frames at least twice as fast as real time
 *             (the page measures the server's real-time factor at 0.08-0.10),
 *             a chunk that long arrives before the audio queued ahead of it
 *             has played out, so playback started on the first chunk never
 *             stalls for want of frames.  With first = 4 it gives 4, 4, 8, 16,
 *             25, the page's example ramp; with first = 1, 1, 1, 2, 4, 8, 16,
 *             25.  (The page names the adaptive mode without defining it; this
 *             doubling rule is the reading taken.)
 */
#define CODEC_SCHEDULE_FIXED 0
#define CODEC_SCHEDULE_RAMP 1
#define CODEC_SCHEDULE_ADAPTIVE 2
typedef struct codec_chunk_schedule {
    int32_t kind;       /* CODEC_SCHEDULE_* */
    int32_t first;      /* FIXED, ADAPTIVE: frames of chunk 0 (>= 1) */
    int32_t steady;     /* frames of the steady chunks (>= 1; 25 on the server) */
    int32_t n_ramp;     /* RAMP: entries of ramp (0..8) */
    int32_t ramp[8];
} codec_chunk_schedule;

CODEC_API int32_t codec_chunk_frames(const codec_chunk_schedule* schedule, int32_t index, int64_t frames_delivered);

/* Host-buffer form: codes_host int32 [B][Q][T_max] and audio_host float
 * [B][T_max * spf] are host memory (page-locked for asynchronous copies).  The
 * call copies the codes to a state-owned device buffer, decodes, copies the
 * audio back and synchronises stream before returning. */
CODEC_API codec_status codec_decode_chunk_host(codec_state_t* state, const int32_t* codes_host,
                                     const int32_t* n_frames, const int32_t* stream_ids, int32_t B,
                                     int32_t T_max, float* audio_host, void* stream);

/*
 * One causal dilated Conv1d on the tensor-core fp16x3 path, outside the
 * decoder: y[t] = bias + sum_j sum_ci W[co][ci][j] a[H + t - (k-1-j) dil][ci],
 * a = Snake_alpha(x) when alpha is given, else x, H = (k-1) dil.  The same
 * operand split, tcgen05 GEMM and chunked accumulation as the decoder's convs;
 * for verification of that kernel and for callers composing their own layers.
 *   x     device float [H + T][Cin], the H history rows first
 *   w     device float [Cout][Cin][k] (PyTorch Conv1d layout)
 *   bias  device float [Cout] or NULL;  alpha device float [Cin] or NULL
 *   y     device float [T][Cout]
 * Uses the state's scratch, so it needs a state of a tensor-core
 * codec (else CODEC_ERR_CONFIG) and is ordered with that state's other work on
 * the same stream.  Requires Cin % 32 == 0, Cout % 16 == 0, T >= 1,
 * 1 <= k <= 16, dilation >= 1, Cin <= 4096 when alpha is given
 * (CODEC_ERR_ARG); (H + T) * Cin and Cout * Cin * k within the scratch the
 * state sized for its decoder (CODEC_ERR_CAPACITY).
 */
CODEC_API codec_status codec_state_conv1d(codec_state_t* state, const float* x, int32_t T, int32_t Cin,
                                          const float* w, const float* bias, const float* alpha, int32_t Cout,
                                          int32_t k, int32_t dilation, float* y, void* stream);

/*
 * codec_state_conv1d without any device allocation, for callers that cannot
 * allocate at the point of use: a real-time audio thread (cudaMalloc can block
 * for an unbounded time and synchronises the device), a host application
 * whose GPU memory is owned by its own pool allocator, an embedding handed
 * only input and output buffers.  The pages have no counterpart of this entry
 * point; it is a service of this library.
 *
 * Same computation, arguments, layouts and argument errors as
 * codec_state_conv1d (checked first), but no codec or state: the caller
 * passes the inputs and the output, and the scratch (operand planes, plan,
 * weight scale, timeout flag) lives in one 32 MiB device array of the library,
 * which every GPU that loads the library keeps until the process exits.
 * Limits: (H + T) * Cin <= 4,194,304 and Cout * Cin * k <= 4,194,304, else
 * CODEC_ERR_CAPACITY; with either error nothing is enqueued.  The first call
 * on a device looks up the array's device address on the current device (no
 * allocation); make that first call before any stream capture.  All calls on
 * a device share the array and it keeps the last call's contents (each call
 * rewrites what it reads, and clears the timeout flag on its stream first):
 * calls that overlap on the GPU, on different streams or threads, race on it.
 */
CODEC_API codec_status codec_conv1d_noalloc(const float* x, int32_t T, int32_t Cin, const float* w,
                                            const float* bias, const float* alpha, int32_t Cout, int32_t k,
                                            int32_t dilation, float* y, void* stream);

/* Whether the last codec_conv1d_noalloc call on the current device gave up on
 * one of the tensor-core kernel's bounded waits (its output is then not
 * valid): *timed_out = 1, else 0.  Synchronises stream first (host-blocking)
 * and allocates nothing.  Errors: CODEC_ERR_NULL, CODEC_ERR_NO_DEVICE,
 * CODEC_ERR_CUDA. */
CODEC_API codec_status codec_conv1d_noalloc_status(int32_t* timed_out, void* stream);

/* Frames decoded and sticky error bits of one slot.  Synchronises stream
 * (host-blocking).  Errors: CODEC_ERR_NULL, CODEC_ERR_ARG, CODEC_ERR_CUDA. */
CODEC_API codec_status codec_state_query(codec_state_t* state, int32_t stream_id, codec_stream_info* info,
                               void* stream);

/* Graph replay (on by default): a decode call whose shape (the per-stream
 * frame counts, T_max) and buffers (codes, audio, pre_tanh) match an earlier
 * call replays that call's captured CUDA graph instead of launching its
 * kernels one by one; a shape is captured the second time it is seen.  Results are the
 * same either way.  enable = 0 turns replay off and frees the graphs (it
 * synchronises the device).  Calls made while codec_profile_begin is active
 * launch directly.  Errors: CODEC_ERR_NULL, CODEC_ERR_CUDA. */
CODEC_API codec_status codec_state_set_graphs(codec_state_t* state, int32_t enable);

/* Bounded waits of the tensor-core kernels for this state's calls (decode and
 * conv1d): every wait gives up after `polls` polls (0: the default, 2^25), the
 * kernel then stops cleanly, and codec_state_query reports
 * CODEC_STREAM_ERR_KERNEL_TIMEOUT until a reset of all slots.  unarrived_wait
 * != 0 exists to verify that path: each GEMM CTA's first epilogue wait then
 * targets a barrier that no role ever arrives on, so it runs out after
 * `polls` polls on any input (results of such calls are not valid).  Drops
 * the captured graphs (synchronises the device).  Errors: CODEC_ERR_NULL,
 * CODEC_ERR_CUDA. */
CODEC_API codec_status codec_state_set_wait_limit(codec_state_t* state, uint32_t polls, int32_t unarrived_wait);

/* Number of stream slots of a state. */
CODEC_API int32_t codec_state_streams(const codec_state_t* state);

/* Number of kernel launches the last decode call enqueued. */
CODEC_API int32_t codec_state_last_launches(const codec_state_t* state);

/* Per-launch timing for measurement.  codec_profile_begin makes later decode
 * calls on this state record a CUDA event pair around every kernel they
 * launch (up to max_records launches; the events are created here, never in
 * a decode call).  codec_profile_end synchronises the stream the calls used,
 * sums the event intervals per kernel kind and stops recording.  Each
 * record also carries the algorithmic work of its launch: useful
 * floating-point operations (2 per multiply-add) and the bytes the operation
 * must move at minimum (inputs read once, outputs written once).  While
 * recording, a call runs the resblocks of each multi-receptive-field block one
 * after the other on the caller's stream (otherwise resblocks 1 and 2 run
 * concurrently with resblock 0 on internal streams), so that no two recorded
 * launches overlap; the results are the same either way. */
typedef enum codec_kernel_kind {
    CODEC_KERNEL_GATHER = 0,
    CODEC_KERNEL_GEMM_SIMT = 1,
    CODEC_KERNEL_GEMM_TC = 2,
    CODEC_KERNEL_OPERAND_PREP = 3,
    CODEC_KERNEL_RMSNORM = 4,
    CODEC_KERNEL_ATTENTION = 5,
    CODEC_KERNEL_FINAL_CONV = 6,
    CODEC_KERNEL_HISTORY = 7,
    CODEC_KERNEL_MRF_SUM = 8,   /* the MRF average of a small call's separately written resblocks */
    CODEC_KERNEL_KINDS = 9
} codec_kernel_kind;

typedef struct codec_kernel_stats {
    int32_t kind;            /* codec_kernel_kind */
    int32_t launches;
    double ms;               /* summed event intervals */
    double flops;            /* summed algorithmic flops */
    double bytes;            /* summed algorithmic bytes */
} codec_kernel_stats;

CODEC_API codec_status codec_profile_begin(codec_state_t* state, int32_t max_records);
/* out: host [CODEC_KERNEL_KINDS]; entry i describes kind i.  Records beyond
 * max_records are dropped (launches still run).  The per-launch records stay
 * readable with codec_profile_launches until the next codec_profile_begin. */
CODEC_API codec_status codec_profile_end(codec_state_t* state, codec_kernel_stats* out, void* stream);

typedef struct codec_launch_record {
    int32_t kind;            /* codec_kernel_kind */
    int32_t reserved;
    double ms, flops, bytes;
} codec_launch_record;

/* The records of the last profiled interval, in launch order: out host
 * [max_out]; *n_out receives the number written.  Call after
 * codec_profile_end. */
CODEC_API codec_status codec_profile_launches(codec_state_t* state, codec_launch_record* out, int32_t max_out,
                                              int32_t* n_out);

/*
 * Streaming iSTFT head: the last step of the iSTFT-head vocoders the pages
 * list (F5-TTS's Vocos, "Vocos -> iSTFT"; CosyVoice2's and Chatterbox's HiFT,
 * "F0 -> NSF source, iSTFT"; Kokoro's iSTFTNet generator, whose iSTFT the Core
 * AI Kokoro note runs as a transposed convolution of stride 5 from 11 channels
 * to 1, i.e. n_fft 20 and hop 5).  Independent of codec_t.
 *
 * A frame holds n_bins = n_fft / 2 + 1 log-magnitudes L[k], then n_bins phases
 * p[k] in radians.  X[k] = min(exp(L[k]), mag_clip) * (cos p[k] + i sin p[k])
 * (no clip when mag_clip <= 0); the frame's signal is the inverse real DFT of
 * X (the imaginary parts of the DC and Nyquist bins are ignored) times the
 * periodic Hann window w[m] = sin^2(pi m / n_fft); frames are overlap-added at
 * hop and the sum is divided by the stationary window-square envelope
 * E[n mod hop] = sum_j w[(n mod hop) + j hop]^2.  Streaming is causal: frames
 * before a stream's start are zero, and frame t completes samples
 * [t hop, (t + 1) hop), so a call of n frames returns n * hop samples; each
 * stream carries its last n_fft / hop - 1 windowed frames.
 *
 * Limits: n_fft even, 4 <= n_fft <= 4096, hop >= 1 dividing n_fft.  Power-of-
 * two n_fft uses a radix-4 (and radix-2) Stockham FFT in shared memory, other sizes a direct DFT.
 */
typedef struct codec_istft_config {
    int32_t n_fft;
    int32_t hop;
    float mag_clip;            /* magnitudes above this are clipped; <= 0: no clip */
    int32_t max_streams;       /* stream slots */
    int32_t max_chunk_frames;  /* frames per stream and call */
} codec_istft_config;

typedef struct codec_istft_s codec_istft_t;

/* All device memory (per-slot carried frames, the per-call frame scratch,
 * the envelope and twiddle tables, the plan) is allocated here on the current
 * device; every slot starts reset.  CODEC_ERR_CONFIG for limits outside the
 * above.  A codec_istft_t is used by one host thread at a time, and its calls
 * go to one stream at a time (they share the plan and the frame scratch). */
CODEC_API codec_status codec_istft_create(const codec_istft_config* cfg, codec_istft_t** out);

/* Synchronises the device, then frees everything. */
CODEC_API void codec_istft_destroy(codec_istft_t* istft);

/* Clears the carried frames of stream_ids (host, n ids; NULL: all slots),
 * stream-ordered on `stream`. */
CODEC_API codec_status codec_istft_reset(codec_istft_t* istft, const int32_t* stream_ids, int32_t n,
                                         void* stream);

/* One chunk for B streams.  spec: device float [B][T_max][2 n_bins] (batch
 * entry b's frames 0 .. n_frames[b] - 1 are read); n_frames: host [B], each in
 * 0 .. T_max; stream_ids: host [B] distinct slots, or NULL for 0 .. B-1;
 * audio: device float [B][T_max hop], entry b's first n_frames[b] hop samples
 * are written.  The caller owns spec and audio and keeps them alive until
 * `stream` passes the call.  Argument errors (B > max_streams, T_max >
 * max_chunk_frames, repeated ids, n_frames out of range) return before
 * anything is enqueued. */
CODEC_API codec_status codec_istft_decode(codec_istft_t* istft, const float* spec, const int32_t* n_frames,
                                          const int32_t* stream_ids, int32_t B, int32_t T_max, float* audio,
                                          void* stream);

/*
 * Harmonic sine source: the hn-NSF excitation of the iSTFT-head vocoders (the
 * Core AI Kokoro note: "har = STFT(SineGen(f0_upsamp(F0)))"; HiFT's "F0 -> NSF
 * source").  Per stream and F0 frame (Hz), held for upp samples:
 * D = rint(min(max(F0, 0), fs / 2) * (2^32 / fs)) is the phase increment per
 * sample in units of 2^-32 cycle (float64 arithmetic, round half to even);
 * the phase P[n] = (P[n - 1] + D) mod 2^32 is an exact integer running sum,
 * carried between calls (0 after reset); output
 * out[n][h - 1] = amplitude * sin(2 pi (h P[n] mod 2^32) / 2^32) for
 * h = 1 .. harmonics where F0 > voiced_threshold, else 0.
 * Limits: 1 <= upp <= 65536, 1 <= harmonics <= 16, sample_rate > 0.
 */
typedef struct codec_sine_config {
    int32_t upp;               /* samples per F0 frame */
    float sample_rate;
    int32_t harmonics;
    float amplitude;
    float voiced_threshold;
    int32_t max_streams;
    int32_t max_chunk_frames;
} codec_sine_config;

typedef struct codec_sine_s codec_sine_t;

/* Allocates the per-slot phases and the per-call plan and frame scratch on
 * the current device, all slots reset.  One host thread and one stream at a
 * time per object. */
CODEC_API codec_status codec_sine_create(const codec_sine_config* cfg, codec_sine_t** out);
CODEC_API void codec_sine_destroy(codec_sine_t* sine);
/* Phases of stream_ids (host, n; NULL: all) back to 0, stream-ordered. */
CODEC_API codec_status codec_sine_reset(codec_sine_t* sine, const int32_t* stream_ids, int32_t n, void* stream);
/* f0: device float [B][T_max] (entry b's first n_frames[b] frames read);
 * n_frames, stream_ids: host [B] (ids distinct, NULL: 0 .. B-1); out: device
 * float [B][T_max upp][harmonics], entry b's first n_frames[b] upp rows
 * written.  Argument errors return before anything is enqueued. */
CODEC_API codec_status codec_sine_decode(codec_sine_t* sine, const float* f0, const int32_t* n_frames,
                                         const int32_t* stream_ids, int32_t B, int32_t T_max, float* out,
                                         void* stream);

/*
 * Streaming analysis STFT (the "STFT" of the same excitation path): frame t
 * of a stream covers its input samples [(t + 1) hop - n_fft, (t + 1) hop)
 * (zeros before the stream's start), times the periodic Hann window
 * w[m] = sin^2(pi m / n_fft); X_t[k] = sum_m w[m] x[m] exp(-2 pi i k m /
 * n_fft), k = 0 .. n_fft / 2.  Every hop of input yields one frame; each
 * stream carries its last n_fft - hop input samples.  Fed to the iSTFT head
 * (as log|X| and arg X) it returns the input delayed by n_fft - hop samples.
 * Limits as for the iSTFT head.
 */
typedef struct codec_stft_config {
    int32_t n_fft;
    int32_t hop;
    int32_t max_streams;
    int32_t max_chunk_frames;  /* hops (frames) per stream and call */
} codec_stft_config;

typedef struct codec_stft_s codec_stft_t;

/* Allocates the per-slot input history (two buffers used in turn), the
 * twiddle table and the plan on the current device, all slots reset.  One
 * host thread and one stream at a time per object. */
CODEC_API codec_status codec_stft_create(const codec_stft_config* cfg, codec_stft_t** out);
CODEC_API void codec_stft_destroy(codec_stft_t* stft);
CODEC_API codec_status codec_stft_reset(codec_stft_t* stft, const int32_t* stream_ids, int32_t n, void* stream);
/* x: device float [B][T_max hop] (entry b's first n_frames[b] hop samples
 * read); n_frames: host [B], hops per entry, 0 .. T_max; stream_ids as above;
 * spec: device float [B][T_max][2 (n_fft / 2 + 1)], per frame the real parts
 * then the imaginary parts; entry b's first n_frames[b] frames written. */
CODEC_API codec_status codec_stft_decode(codec_stft_t* stft, const float* x, const int32_t* n_frames,
                                         const int32_t* stream_ids, int32_t B, int32_t T_max, float* spec,
                                         void* stream);

/*
 * Streaming Vocos-style generator in front of the iSTFT head (vox, "How each
 * model runs": F5-TTS ends in "Vocos -> iSTFT"), causal like the decoder:
 *   h = LayerNorm(conv_k(mel) + b)                          (embedding, causal)
 *   per block: h = h + gamma * (W2 GELU(W1 LayerNorm(dwconv_k(h) + b_dw) + b1) + b2)
 *   spec = W_head LayerNorm(h) + b_head: n_fft / 2 + 1 log-magnitudes, then
 *   as many phases; audio = the streaming iSTFT head above (mag_clip).
 * LayerNorm over the channels with biased variance, eps inside the root;
 * GELU in its erf form; dwconv a per-channel causal conv.  Each stream carries
 * the embedding conv's last k - 1 mel rows, each block's last k - 1 input rows
 * and the head's frames, so chunked decoding equals a full decode.  The
 * pointwise layers run on the tcgen05 fp16x3 path when precision asks for it
 * and their channel counts allow (the layer scale folded into W2 and b2); the
 * rest in fp32.
 */
typedef struct codec_vocos_config {
    int32_t n_mels, d, ffn, layers;   /* multiples of 4; d <= 1024 */
    int32_t k;                        /* embedding and depthwise kernel, 1..16 */
    int32_t n_fft, hop;               /* as codec_istft_config */
    float ln_eps, mag_clip;
    int32_t max_streams, max_chunk_frames, max_batch_frames;
    int32_t precision;                /* codec_precision */
} codec_vocos_config;

typedef struct codec_vocos_s codec_vocos_t;

/* Weight blob (fp32, PyTorch layouts) in this order: embedding conv [d][n_mels][k],
 * bias [d]; LayerNorm gain, bias [d]; per block: depthwise taps [d][1][k], bias [d],
 * LayerNorm gain, bias [d], W1 [ffn][d], b1 [ffn], W2 [d][ffn], b2 [d], layer scale
 * [d]; final LayerNorm gain, bias [d]; head [n_fft + 2][d], bias [n_fft + 2].
 * Returns its length in floats, or -1 for an invalid config. */
CODEC_API int64_t codec_vocos_weight_floats(const codec_vocos_config* cfg);

/* Allocates everything on the current device (slots reset).  One host thread
 * and one stream at a time per object.  Errors as codec_create. */
CODEC_API codec_status codec_vocos_create(const codec_vocos_config* cfg, const float* weights, int64_t n_floats,
                                          codec_vocos_t** out);
CODEC_API void codec_vocos_destroy(codec_vocos_t* vocos);
CODEC_API codec_status codec_vocos_reset(codec_vocos_t* vocos, const int32_t* stream_ids, int32_t n, void* stream);

/* mel: device float [B][T_max][n_mels] (entry b's first n_frames[b] frames);
 * n_frames, stream_ids: host [B] (ids distinct, NULL: 0 .. B-1); audio: device
 * float [B][T_max hop], entry b's first n_frames[b] hop samples written.
 * Argument errors (as codec_decode_chunk) return before anything is enqueued. */
CODEC_API codec_status codec_vocos_decode(codec_vocos_t* vocos, const float* mel, const int32_t* n_frames,
                                          const int32_t* stream_ids, int32_t B, int32_t T_max, float* audio,
                                          void* stream);

/* Static description of a status code. */
CODEC_API const char* codec_status_string(codec_status status);

#ifdef __cplusplus
}
#endif

#endif /* GB300_CODEC_H */
