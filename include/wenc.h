/*
 * wenc.h -- C ABI of libwenc.so: the Whisper encoder's pre-LayerNorm transformer
 * blocks, GPU-resident on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the encoder block of the three pages this library follows:
 *   "inferencelayer 0.2.4 src/whisper_gpu.rs" (WhisperEncoderGpu::forward, the
 *     VANILLA_ATTN and LN_SRC shaders),
 *   "turbospark-runtime 0.3.0 src/whisper/metal.rs" (EncLayerGpu, encode_partial,
 *     encode_layer),
 *   "oxinfer 0.0.5 src/whisper/model.rs" (WhisperModel::encode, make_lin, Precision).
 * Per block:  x += Wo . Attn(LN1(x) Wq^T + bq, LN1(x) Wk^T, LN1(x) Wv^T + bv) + bo
 *             x += W2 . GELU_erf(LN2(x) W1^T + b1) + b2
 * then, optionally, a final LayerNorm. Attention is non-causal scaled-dot attention
 * (scale hd^-0.5) over the whole window, with no mask and no positional term.
 *
 * Conventions for every entry point:
 *  - All pointers are DEVICE pointers unless stated otherwise; sizes are element counts.
 *  - Activations are row-major [rows, width]; a window of T frames occupies T consecutive
 *    rows; head h of an attention operand sits in columns h*hd .. h*hd+hd-1.
 *  - Weight matrices are [n_out, n_in] row-major (PyTorch layout); y = x W^T + b.
 *  - bf16 buffers are raw bfloat16 bit patterns (uint16_t).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *    Entry points marked "stream-ordered" do not synchronise the host and allocate nothing,
 *    so a call can be captured into a CUDA graph (make one ordinary call first: the first
 *    call on a device does one-time set-up); a replay gives the bits of an eager call.
 *  - Separate handles may be used from separate host threads at the same time. Calls on one
 *    handle share its workspace and must be ordered by the caller (one stream, or events).
 *  - Argument errors are reported synchronously as a status; the message is available
 *    from wenc_last_error() on the same host thread. Nothing aborts the process.
 *  - Device-side waits are bounded (about one second); a wait that runs out records
 *    WENC_ERR_DEVICE_TIMEOUT in a device error word instead of hanging the GPU. It is
 *    reported by wenc_sync_status() and by the next wenc_forward* call on that handle.
 *  - The bf16 contractions with output widths that are multiples of 256 run on pairs of SMs
 *    (thread-block clusters of two). Setting the environment variable WENC_GEMM_PAIR=0 before
 *    the first call keeps them on single SMs. The results are the same bits either way; the
 *    variable exists for performance comparisons.
 */
#ifndef WENC_H
#define WENC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WENC_API __attribute__((visibility("default")))
#else
#define WENC_API
#endif

typedef struct CUstream_st* wenc_stream_t; /* same type as cudaStream_t */

typedef enum {
  WENC_OK = 0,
  WENC_ERR_INVALID_ARG = 1,     /* null pointer, bad size, misaligned buffer */
  WENC_ERR_UNSUPPORTED = 2,     /* a shape or mode this build does not implement (e.g. hd != 64) */
  WENC_ERR_OOM = 3,             /* device allocation failed (wenc_create, wenc_set_stem, wenc_set_cross_kv) */
  WENC_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed; see wenc_last_error() */
  WENC_ERR_DEVICE_TIMEOUT = 5   /* a bounded device-side wait ran out (pipeline stalled) */
} wenc_status;

/* Storage type of the weight matrices handed to wenc_create. Norm parameters and
 * biases are always float32 ("Norms, biases and positions always stay f32",
 * oxinfer src/whisper/model.rs, Precision). */
typedef enum { WENC_DTYPE_F32 = 0, WENC_DTYPE_BF16 = 1 } wenc_dtype;

/* Arithmetic of the contractions. In both, LayerNorm statistics, softmax, GELU, the
 * accumulators and the residual stream are fp32.
 * BF16: bf16 operands on the tensor cores (kind::f16); matrices rounded to bf16 at create
 *   (nearest-even), activations between kernels (LN output, Q/K/V, P, attention output,
 *   fc1 output) stored as bf16.
 * TF32: TF32 operands on the tensor cores (kind::tf32: 10 explicit mantissa bits, fp32
 *   exponent range); matrices kept as fp32 rounded to TF32 at create (nearest, ties away
 *   from zero; bf16 matrices are widened exactly), activations between kernels stored as
 *   fp32 rounded to TF32 by the kernel that writes them. Twice the operand bytes and half
 *   the tensor-core rate of BF16, for about sixteen times smaller operand rounding
 *   (oxinfer src/whisper/model.rs, Precision: F32 beside Bf16). */
typedef enum { WENC_PREC_BF16 = 0, WENC_PREC_TF32 = 1 } wenc_precision;

/* Epilogues of wenc_linear (the fused forms the block uses). */
typedef enum {
  WENC_EPI_BIAS_BF16 = 0,       /* out(bf16) = A W^T + bias                         (QKV)   */
  WENC_EPI_BIAS_GELU_BF16 = 1,  /* out(bf16) = GELU_erf(A W^T + bias)               (fc1)   */
  WENC_EPI_BIAS_RESID_F32 = 2   /* out(f32)  = resid + A W^T + bias (resid may == out) (out-proj, fc2) */
} wenc_epilogue;

typedef struct {
  int n_layers;      /* >= 1 */
  int d_model;       /* = n_heads * head_dim; a multiple of 128 (384, 512, 768, 1280, ...) */
  int n_heads;       /* >= 1 */
  int head_dim;      /* must be 64 */
  int ffn_dim;       /* a multiple of 128 */
  int seq_len;       /* frames per window, 1..4096 (1500 for Whisper's 30 s window) */
  int max_batch;     /* windows per call, >= 1; sizes the workspace */
  int final_ln;      /* nonzero: apply the final LayerNorm after the last block */
  float ln_eps;      /* LayerNorm epsilon (1e-5 on all three pages) */
  int weight_dtype;  /* wenc_dtype of the matrices in wenc_layer_weights */
  int precision;     /* wenc_precision: WENC_PREC_BF16 or WENC_PREC_TF32 */
} wenc_config;

/* One block's parameters, as DEVICE pointers owned by the caller. Matrices are
 * [n_out, n_in] row-major in config.weight_dtype: wq, wk, wv, wo [d, d]; w1 [f, d];
 * w2 [d, f]. Vectors are float32: ln*_w, ln*_b, bq, bv, bo [d]; b1 [f]; b2 [d].
 * bk must be NULL: the K projection has no bias (turbospark-runtime EncLayerGpu). */
typedef struct {
  const float* ln1_w; const float* ln1_b;
  const void* wq; const float* bq;
  const void* wk; const float* bk;
  const void* wv; const float* bv;
  const void* wo; const float* bo;
  const float* ln2_w; const float* ln2_b;
  const void* w1; const float* b1;
  const void* w2; const float* b2;
} wenc_layer_weights;

/* The convolutional stem in front of the blocks (optional; see wenc_set_stem). Device
 * pointers owned by the caller. Matrices in config.weight_dtype with the checkpoint layout
 * [C_out, C_in, 3]; vectors float32. */
typedef struct {
  int n_mels;             /* mel bands of the input: a multiple of 8, 8..1024 (80; 128 for large-v3) */
  const void* conv1_w;    /* [d, n_mels, 3]: kernel 3, stride 1, padding 1 */
  const float* conv1_b;   /* [d] */
  const void* conv2_w;    /* [d, d, 3]: kernel 3, stride 2, padding 1 */
  const float* conv2_b;   /* [d] */
  const float* positions; /* [seq_len, d]: row t is added to output position t after conv2's GELU */
} wenc_stem_weights;

typedef struct wenc wenc; /* opaque handle */

/* wenc_create -- validate `cfg`, pack the weights into library-owned device memory
 * (matrices rounded to bf16, nearest-even, as oxinfer make_lin does for Precision::Bf16,
 * or kept as fp32 rounded to TF32 when cfg->precision is WENC_PREC_TF32; Q/K/V packed into one [3d, d] matrix with a [3d] bias whose K slot is zero, the
 * layout of turbospark-runtime DecLayerGpu::self_qkv_w), and allocate the activation
 * workspace for cfg->max_batch windows (all scratch sized once, as turbospark-runtime's
 * engine does at open). `layers` holds cfg->n_layers entries; lnf_w/lnf_b [d] are read
 * only when cfg->final_ln is set (may be NULL otherwise). The caller's buffers may be
 * freed once this returns: it synchronises `stream` before returning.
 * Errors: INVALID_ARG (null/inconsistent sizes, bk != NULL, `stream` being captured into a
 * CUDA graph: refused before it is touched, so the capture stays intact), UNSUPPORTED (hd != 64,
 * d or f not a multiple of 128, seq_len > 4096), OOM (nothing stays allocated), CUDA. On error
 * *out is NULL. */
WENC_API wenc_status wenc_create(const wenc_config* cfg, const wenc_layer_weights* layers,
                        const float* lnf_w, const float* lnf_b, wenc_stream_t stream,
                        wenc** out);

/* wenc_forward -- hidden_out = Encoder(hidden_in), both float32 [B, seq_len, d_model],
 * caller-owned, hidden_in == hidden_out allowed. 1 <= B <= max_batch. Stream-ordered.
 * One call runs every block and, if configured, the final LayerNorm
 * (inferencelayer WhisperEncoderGpu::forward; oxinfer WhisperModel::encode). */
WENC_API wenc_status wenc_forward(wenc* h, const float* hidden_in, float* hidden_out, int B,
                         wenc_stream_t stream);

/* wenc_forward_layers -- run blocks first .. first+count-1 only, then the final
 * LayerNorm iff apply_final_ln (and the handle has one). The per-layer bisection of
 * turbospark-runtime encode_partial(stop_after). Same buffers and rules as wenc_forward;
 * count may be 0 (then only the final LN, or a copy, runs). Stream-ordered. */
WENC_API wenc_status wenc_forward_layers(wenc* h, const float* hidden_in, float* hidden_out, int B,
                                int first, int count, int apply_final_ln, wenc_stream_t stream);

/* wenc_set_stem -- attach the convolutional stem to a handle (turbospark-runtime
 * encode_partial's conv front end; oxinfer WhisperModel::encode):
 *   h = GELU_erf(conv1(mel)),  x = GELU_erf(conv2(h)) + positions,
 * conv1 kernel 3 / stride 1 / padding 1 (n_mels -> d over 2*seq_len frames), conv2 kernel 3 /
 * stride 2 / padding 1 (d -> d, 2*seq_len -> seq_len positions). Packs the weights into
 * library-owned memory in the handle's precision (each convolution runs as one tensor-core GEMM
 * over the unfolded signal, weights reordered to [C_out, 3*C_in]) and allocates the stem's
 * workspace for cfg.max_batch windows. A second call replaces the first. Synchronises `stream`
 * before returning; the caller's buffers may then be freed.
 * Errors: INVALID_ARG (NULL pointers, n_mels not a multiple of 8 or outside 8..1024, `stream`
 * being captured), OOM (the handle keeps working without a stem; an earlier stem is gone), CUDA. */
WENC_API wenc_status wenc_set_stem(wenc* h, const wenc_stem_weights* w, wenc_stream_t stream);

/* wenc_stem -- hidden_out = stem(mel): mel float32 [B, 2*seq_len, n_mels] (time-major log-mel
 * frames, caller-owned), hidden_out float32 [B, seq_len, d]. 1 <= B <= max_batch; buffers
 * 16-byte aligned; needs wenc_set_stem first (else INVALID_ARG). Stream-ordered, 4 launches. */
WENC_API wenc_status wenc_stem(wenc* h, const float* mel, float* hidden_out, int B, wenc_stream_t stream);

/* wenc_encode -- the whole encoder from log-mel frames: the stem, every block and (if
 * configured) the final LayerNorm. mel as for wenc_stem; hidden_out float32 [B, seq_len, d].
 * The launch-event hook of wenc_set_launch_events covers all wenc_encode_launches() launches. */
WENC_API wenc_status wenc_encode(wenc* h, const float* mel, float* hidden_out, int B, wenc_stream_t stream);

/* wenc_encode_launches -- kernel launches of one wenc_encode call (-1 without a stem). */
WENC_API int wenc_encode_launches(const wenc* h);

/* wenc_set_cross_kv -- attach the decoder's cross-attention K/V weights (n_dec_layers >= 1;
 * wk[l], wv[l]: [d, d] in config.weight_dtype, [n_out, n_in]; bv[l]: [d] float32; all device
 * pointers owned by the caller). They are packed into one [2 n_dec d, d] matrix in the handle's
 * precision (K of layer l at rows 2l*d.., V at (2l+1)*d..; K has no bias, as in
 * turbospark-runtime build_cross_caches). A second call replaces the first. Synchronises
 * `stream` before returning. Errors: INVALID_ARG (NULL pointers, n_dec_layers < 1, `stream` being
 * captured), OOM (the handle keeps working without cross K/V weights; earlier ones are gone), CUDA. */
WENC_API wenc_status wenc_set_cross_kv(wenc* h, int n_dec_layers, const void* const* wk, const void* const* wv,
                                       const float* const* bv, wenc_stream_t stream);

/* wenc_cross_kv -- every decoder layer's cross-attention keys and values over an encoder
 * output (inferencelayer's cross K/V precompute; turbospark-runtime build_cross_caches):
 * K_l = enc_out Wk_l^T, V_l = enc_out Wv_l^T + bv_l. enc_out float32 [B, seq_len, d];
 * kv_out [2 n_dec][B * seq_len][d], plane 2l = K_l and 2l+1 = V_l, in the operand format of the
 * handle's precision (bf16 for WENC_PREC_BF16, float32 rounded to TF32 for WENC_PREC_TF32),
 * caller-owned. 1 <= B <= max_batch; buffers 16-byte aligned; needs wenc_set_cross_kv first.
 * Stream-ordered, 2 launches (the operand cast of enc_out, one GEMM over all layers). */
WENC_API wenc_status wenc_cross_kv(wenc* h, const float* enc_out, void* kv_out, int B, wenc_stream_t stream);

/* wenc_forward_launches -- number of kernel launches one wenc_forward_layers call with
 * these arguments makes (for launch accounting). Returns -1 on bad arguments. */
WENC_API int wenc_forward_launches(const wenc* h, int first, int count, int apply_final_ln);

/* wenc_set_launch_events -- optional timing hook. When `events` is non-NULL, the next
 * forward call records events[0] before its first launch and events[i+1] after launch i
 * (each a cudaEvent_t created by the caller), for n_events >= launches + 1; the hook
 * then clears itself. kinds (may be NULL) receives, per launch, 0 = LayerNorm,
 * 1 = QKV GEMM, 2 = attention, 3 = out-proj GEMM, 4 = fc1 GEMM, 5 = fc2 GEMM,
 * 6 = final LayerNorm, 7 = copy, 8 = attention split-key merge (small batches only),
 * 9 = stem unfold, 10 = stem conv1 GEMM, 11 = stem conv2 GEMM (wenc_stem, wenc_encode),
 * 12 = cross K/V operand cast, 13 = cross K/V GEMM (wenc_cross_kv), 14 = row statistics of the
 * first block's input (BF16 precision, which folds LN1 into the QKV GEMM: kind 0 is then LN2). */
WENC_API wenc_status wenc_set_launch_events(wenc* h, void* const* events, int n_events, int* kinds);

/* wenc_attention -- out = softmax(q k^T * hd^-0.5) v per (window, head), non-causal,
 * over all T keys of each window (inferencelayer VANILLA_ATTN; turbospark-runtime
 * encode_layer's per-head score planes, row softmax and PV).
 * q, k, v, out: bf16 [B, T, H, hd] contiguous (row stride H*hd), caller-owned; the
 * softmax and accumulation are fp32, the output rounded to bf16. hd must be 64;
 * 1 <= T <= 1<<20; B, H >= 1. Buffers must be 16-byte aligned. Stream-ordered.
 * A stalled device wait is recorded in the library's global error word
 * (see wenc_sync_status(NULL)). */
WENC_API wenc_status wenc_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           uint16_t* out, int B, int T, int H, int hd, wenc_stream_t stream);

/* wenc_attention_static -- the attention of wenc_attention (same arguments, layouts, rounding
 * and error reporting) for callers that must not allocate device memory: a host that only lends
 * memory from its own fixed pool, a runtime that forbids allocation while it serves requests, or
 * code that cannot afford the device synchronisation an allocation may cause. The pages have no
 * counterpart to this entry point. The keys of each query pair are split among several CTAs and
 * the partial results are merged by a second kernel; those partial results live in a static
 * device buffer that belongs to the library image (wenc_attention_static_capacity() bytes,
 * 16 MiB, held on every GPU that loads the library until the process exits) instead of memory
 * allocated here. The call allocates nothing. Limits: it needs (splits * B * H * T) * 264 bytes
 * of that buffer, at least two splits when T > 128; larger problems are rejected with
 * WENC_ERR_INVALID_ARG and a message naming the sizes (wenc_attention handles any size).
 * The first call on each device looks up the buffer's device address (cudaGetSymbolAddress
 * with that device current); make that first call before any stream capture. Every call
 * shares the one buffer: calls whose work overlaps on the GPU (other streams, other host
 * threads) race and must be ordered by the caller. Nothing in the buffer needs clearing: each
 * call writes every partial result it later reads. Stream-ordered; hd must be 64. */
WENC_API wenc_status wenc_attention_static(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                           uint16_t* out, int B, int T, int H, int hd, wenc_stream_t stream);

/* wenc_attention_static_capacity -- bytes of the static buffer wenc_attention_static uses. */
WENC_API size_t wenc_attention_static_capacity(void);

/* wenc_layernorm -- y = (x - mean) / sqrt(var + eps) * w + b per row of x float32
 * [rows, d] (biased variance; inferencelayer LN_SRC). out_format: 0 = float32, 1 = bf16
 * (the cast that feeds a BF16 GEMM), 2 = float32 rounded to TF32 (feeds a TF32 GEMM);
 * anything else is INVALID_ARG. d a multiple of 128, <= 2048. Stream-ordered. */
WENC_API wenc_status wenc_layernorm(const float* x, const float* w, const float* b, void* y, int rows,
                           int d, float eps, int out_format, wenc_stream_t stream);

/* wenc_linear -- one contraction of the block with a fused epilogue (see wenc_epilogue):
 * A bf16 [M, K], W bf16 [N, K] (K-major, PyTorch layout), bias float32 [N], resid/out
 * [M, N] (bf16 or f32 per the epilogue). N a multiple of 128, K a multiple of 64, M >= 1.
 * Buffers 16-byte aligned. Stream-ordered. The matmul_bias
 * step of turbospark-runtime encode_layer with its add / gelu_erf passes fused in. */
WENC_API wenc_status wenc_linear(const uint16_t* A, const uint16_t* W, const float* bias,
                        const float* resid, void* out, int M, int N, int K, int epilogue,
                        wenc_stream_t stream);

/* wenc_linear_tf32 -- the contraction of wenc_linear in the TF32 precision: A float32
 * [M, K], W float32 [N, K], both read by the tensor cores as TF32 (pass values already
 * rounded to TF32 for round-to-nearest; other low mantissa bits are not used as such), fp32
 * accumulation. Epilogues as wenc_epilogue, except that WENC_EPI_BIAS_BF16 and
 * WENC_EPI_BIAS_GELU_BF16 write float32 rounded to TF32 instead of bf16; out is float32
 * [M, N]. N a multiple of 128, K a multiple of 32, M >= 1; buffers 16-byte aligned.
 * Stream-ordered; errors as wenc_linear. */
WENC_API wenc_status wenc_linear_tf32(const float* A, const float* W, const float* bias,
                                      const float* resid, float* out, int M, int N, int K, int epilogue,
                                      wenc_stream_t stream);

/* wenc_attention_tf32 -- the attention of wenc_attention in the TF32 precision: q, k, v, out
 * float32 [B, T, H, hd] contiguous, caller-owned. Q K^T and P V run on the tensor cores with
 * TF32 operands (q, k, v read as TF32: pass values already rounded to TF32), the
 * probabilities are rounded to TF32 before the PV product, softmax and accumulation are fp32,
 * and the output is float32 rounded to TF32. hd must be 64; 1 <= T <= 1<<20; B, H >= 1.
 * Buffers 16-byte aligned. Stream-ordered; a stalled device wait is recorded as for
 * wenc_attention. */
WENC_API wenc_status wenc_attention_tf32(const float* q, const float* k, const float* v, float* out,
                                         int B, int T, int H, int hd, wenc_stream_t stream);

/* wenc_set_device_alloc_limit -- test hook for the out-of-memory path (the pages have no
 * counterpart). Caps the device memory the library holds in its handles' arenas (weights,
 * workspace, stem, cross K/V) at `bytes`; an allocation that would exceed the cap fails as if
 * cudaMalloc had run out, so wenc_create, wenc_set_stem and wenc_set_cross_kv return
 * WENC_ERR_OOM and release what they allocated. 0 removes the cap (the default). Process-wide;
 * not meant for concurrent use with other threads creating handles. */
WENC_API void wenc_set_device_alloc_limit(size_t bytes);

/* wenc_device_bytes_held -- bytes of device memory the library holds in live arenas (all
 * handles of the process), for leak checks. */
WENC_API size_t wenc_device_bytes_held(void);

/* wenc_selftest_wait_timeout -- exercises the failure path of the bounded device waits
 * (the pages have no counterpart). Launches one CTA
 * that waits on an mbarrier nothing ever arrives on, with the same bounded wait every kernel
 * uses: after about one second the wait gives up, records WENC_ERR_DEVICE_TIMEOUT (site 99)
 * in the handle-less device error word and the kernel returns; no trap, the context stays
 * usable. Stream-ordered; read the outcome with wenc_sync_status(NULL). */
WENC_API wenc_status wenc_selftest_wait_timeout(wenc_stream_t stream);

/* wenc_selftest_gemm_pair_abort -- exercises the failure path of the CTA-pair GEMM (the pages
 * have no counterpart). Runs out = bf16(A W^T + bias) (A bf16 [M, K], W bf16 [N, K], bias f32
 * [N], out bf16 [M, N], device pointers, 16-byte aligned; N a multiple of 256, K of 64) on CTA
 * pairs, with the odd CTA of every pair giving up after `stop_after` k-block stages as if one of
 * its waits had run out. The even CTA's waits for the missing data then run out too (about a
 * second); the pair drains every copy that may be in flight, in order, before either CTA
 * exits, and WENC_ERR_DEVICE_TIMEOUT is recorded (site 31, or the site of the even CTA's wait)
 * in the handle-less device error word; no trap, the context stays usable and `out` holds no
 * defined values. Stream-ordered; read the outcome with wenc_sync_status(NULL).
 * WENC_ERR_UNSUPPORTED when the CTA-pair form is switched off (WENC_GEMM_PAIR=0). */
WENC_API wenc_status wenc_selftest_gemm_pair_abort(const uint16_t* A, const uint16_t* W, const float* bias,
                                                   uint16_t* out, int M, int N, int K, int stop_after,
                                                   wenc_stream_t stream);

/* wenc_selftest_attention_abort -- exercises the failure path of the attention kernel (the pages
 * have no counterpart). Runs the attention of wenc_attention (same arguments and layouts; no key
 * splits) with its TMA producer giving up after `stop_after` K tiles, as if one of its waits had
 * run out. The MMA and softmax warps then see the CTA's abort flag and stop, the producer drains
 * the copies it issued, every MMA completes before TMEM is freed, and WENC_ERR_DEVICE_TIMEOUT
 * (site 31) is recorded in the handle-less device error word. There is no trap, the context
 * stays usable, and `out` holds no defined values. Stream-ordered; read the outcome with
 * wenc_sync_status(NULL). */
WENC_API wenc_status wenc_selftest_attention_abort(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                                   uint16_t* out, int B, int T, int H, int stop_after,
                                                   wenc_stream_t stream);

/* wenc_selftest_gemm_schedule -- host only, no device work: replays how a contraction of
 * M x N output elements divides its tiles among the units of one launch (single CTAs on
 * 128-row tiles when pair is 0, CTA pairs on 256 x 256 tiles when pair is 1), through the same
 * schedule code the GEMM kernel runs, for a launch of at most max_units units (the SM count, or
 * the number of pairs that fit). cover[2t + h] counts how often column half h of tile t is
 * computed (cover_len >= 2 x tiles); unit_halves[u] (max_units entries, may be NULL) is the
 * number of half tiles unit u computes; *units and *halves receive the launch size and whether
 * its last wave runs as half-width units. Returns WENC_ERR_INVALID_ARG for an unsupported
 * shape or a short cover array. */
WENC_API wenc_status wenc_selftest_gemm_schedule(int M, int N, int pair, int max_units, int* cover, int cover_len,
                                                 int* unit_halves, int* units, int* halves);

/* wenc_sync_status -- synchronise the device and read the device error word of `h`
 * (or, when h is NULL, the word shared by the handle-less entry points), clearing it.
 * Returns WENC_OK, WENC_ERR_DEVICE_TIMEOUT or WENC_ERR_CUDA. */
WENC_API wenc_status wenc_sync_status(wenc* h);

/* wenc_destroy -- free everything the handle owns (synchronises the device first).
 * NULL is a no-op. */
WENC_API void wenc_destroy(wenc* h);

/* wenc_last_error -- message for the last non-OK status returned on this host thread
 * ("" if none). The pointer stays valid until the next call on this thread. */
WENC_API const char* wenc_last_error(void);

/* wenc_version -- "wenc <major>.<minor> sm_103a". */
WENC_API const char* wenc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* WENC_H */
