// api.cu -- the C ABI of libwenc.so: argument checking, weight packing, workspace,
// tensor maps and the per-block launch sequence. Every step of the computation runs in
// the kernels of ln.cu, gemm.cu and attn.cu; this file only prepares and orders them.
//
// Block order (turbospark-runtime 0.3.0 src/whisper/metal.rs, encode_layer; inferencelayer
// 0.2.4 src/whisper_gpu.rs, WhisperEncoderGpu::forward; oxinfer 0.0.5 src/whisper/model.rs,
// WhisperModel::encode), with each add/activation folded into the producing kernel:
//   LN1(x) -> xn (bf16) ; QKV = xn Wqkv^T + [bq;0;bv] ; o = Attn(QKV)
//   x = x + o Wo^T + bo ; LN2(x) -> xn ; u = GELU(xn W1^T + b1) ; x = x + u W2^T + b2
// and the final LayerNorm into the caller's output.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "launch.h"
#include "ptx.cuh"
#include "wenc.h"

namespace {

thread_local std::string g_last_error;

wenc_status fail(wenc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

wenc_status cuda_fail(cudaError_t e, const char* what) {
  return fail(WENC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_device_accessible(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// Device error word shared by the handle-less entry points.
__device__ uint32_t g_device_error_word;

uint32_t* global_error_word(std::string* why) {
  // per-device cache; host threads that race here store the same address
  static std::atomic<uint32_t*> addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *why = "no current CUDA device";
    return nullptr;
  }
  uint32_t* a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_device_error_word);
    if (e != cudaSuccess) {
      *why = std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
      return nullptr;
    }
    a = static_cast<uint32_t*>(p);
    addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

bool device_is_sm103(std::string* why) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *why = "no CUDA device";
    return false;
  }
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    char b[128];
    snprintf(b, sizeof(b), "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    *why = b;
    return false;
  }
  return true;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// One CTA waits on a barrier that nothing arrives on; the bounded wait gives up, records the
// timeout in the error word and the kernel returns normally.
__global__ void stall_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    wenc_dev::mbar_init(wenc_dev::smem_u32(&bar), 1);
    abort_flag = 0u;
    wenc_dev::fence_barrier_init();
  }
  __syncthreads();
  const wenc_dev::WaitCtx wc{&abort_flag, err};
  wenc_dev::mbar_wait(wenc_dev::smem_u32(&bar), 0, wc, 99);
}

}  // namespace

namespace wenc_host {

// One 128-byte-swizzled tiled map of rank 2 or 3 (dims[0] innermost).
static bool make_tmap(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, const void* base, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, std::string* why) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char b[160];
    snprintf(b, sizeof(b), "cuTensorMapEncodeTiled(rank %u, %llu x %llu) failed with %d", rank,
             (unsigned long long)dims[0], (unsigned long long)dims[1], static_cast<int>(r));
    *why = b;
    return false;
  }
  return true;
}

bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                       uint32_t box_inner, uint32_t box_outer, std::string* why) {
  const cuuint64_t dims[2] = {inner, outer}, strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, why);
}

bool make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                      uint32_t box_inner, uint32_t box_outer, std::string* why) {
  const cuuint64_t dims[2] = {inner, outer}, strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, why);
}

bool make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t dim1, uint64_t dim2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box_inner, uint32_t box1,
                       std::string* why) {
  const cuuint64_t dims[3] = {inner, dim1, dim2}, strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box_inner, box1, 1};
  return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, why);
}

bool make_tmap_3d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t dim1, uint64_t dim2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box_inner, uint32_t box1,
                      std::string* why) {
  const cuuint64_t dims[3] = {inner, dim1, dim2}, strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box_inner, box1, 1};
  return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, why);
}

}  // namespace wenc_host

// ================================================================ the handle
struct wenc {
  wenc_config cfg;
  int device = 0;
  int num_sms = 1;
  bool tf32 = false;  // precision WENC_PREC_TF32: fp32 (TF32-rounded) matrices and activations
  size_t esz = 2;     // bytes per matrix / GEMM-operand element: 2 (bf16) or 4 (fp32)
  struct Layer {
    void *wqkv, *wo, *w1, *w2;  // [n_out, n_in], bf16 or TF32-rounded fp32
    float *ln1_w, *ln1_b, *bqkv, *bo, *ln2_w, *ln2_b, *b1, *b2;
    // BF16 precision: LN1 is folded into Wqkv (wqkv and bqkv hold the folded forms) and this
    // holds the row sums of the folded matrix; null for TF32
    float* cs_qkv = nullptr;
    CUtensorMap tm_wqkv, tm_wo, tm_w1, tm_w2;
    CUtensorMap tm_wqkv_h, tm_wo_h, tm_w1_h, tm_w2_h;  // the same with half-height boxes
  };
  std::vector<Layer> layers;
  float* lnf_w = nullptr;
  float* lnf_b = nullptr;
  int bn_qkv = 0, bn_o = 0, bn_1 = 0, bn_2 = 0;
  // workspace (rows = max_batch * seq_len)
  float* x = nullptr;
  void *xn = nullptr, *qkv = nullptr, *o = nullptr, *u = nullptr;  // element size esz
  CUtensorMap tm_xn, tm_o, tm_u, tm_q, tm_kv;
  int attn_splits = 1;            // key splits of the attention (1 = none), fixed at create
  float2* stats = nullptr;        // BF16: row segment statistics of the residual stream (workspace)
  int seg_w = 0;                  // their segment width
  float* part_o = nullptr;        // split-key partial numerators (workspace)
  float2* part_ml = nullptr;      // split-key (max, sum) pairs (workspace)
  void* weight_arena = nullptr;
  void* work_arena = nullptr;
  size_t weight_bytes = 0, work_bytes = 0, stem_bytes = 0, cross_bytes = 0;  // sizes of the four arenas
  uint32_t* err_host = nullptr;  // mapped pinned word: the device writes, the host reads without a sync
  uint32_t* err_dev = nullptr;
  // timing hook (one call)
  std::vector<cudaEvent_t> events;
  int* kinds = nullptr;
  // convolutional stem (wenc_set_stem); weights and workspace in one arena
  bool has_stem = false;
  int n_mels = 0, kp1 = 0, bn_stem = 0;
  void* stem_arena = nullptr;
  void *wc1 = nullptr, *wc2 = nullptr;  // [d, kp1], [d, 3d] in the operand format
  float *cb1 = nullptr, *cb2 = nullptr, *pos = nullptr;
  void *a1 = nullptr, *h1 = nullptr, *a2 = nullptr;  // unfolded mel, conv1 output, unfolded conv1 output
  CUtensorMap tm_a1, tm_wc1, tm_a2, tm_wc2, tm_wc1_h, tm_wc2_h;
  // decoder cross K/V weights (wenc_set_cross_kv): [2 n_dec d, d] operand format, bias [2 n_dec d]
  int n_dec = 0, bn_cross = 0;
  void* cross_arena = nullptr;
  void* wx = nullptr;
  float* bx = nullptr;
  CUtensorMap tm_wx, tm_wx_h;
};

namespace {

// Device memory the library holds (its handles' arenas), and an optional cap on it that a test
// sets to make an allocation fail as if the device had run out (wenc_set_device_alloc_limit).
std::atomic<size_t> g_dev_held{0};
std::atomic<size_t> g_dev_limit{0};  // 0: no cap

cudaError_t dev_alloc(void** p, size_t bytes) {
  *p = nullptr;
  const size_t cap = g_dev_limit.load();
  if (cap != 0 && g_dev_held.load() + bytes > cap) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    return e;
  }
  g_dev_held += bytes;
  return cudaSuccess;
}

void dev_free(void*& p, size_t& bytes) {
  if (!p) return;
  cudaFree(p);
  g_dev_held -= bytes;
  p = nullptr;
  bytes = 0;
}

// Entry points that synchronise their stream (create, set_stem, set_cross_kv) cannot run while
// it is being captured into a CUDA graph: refuse such a stream before touching it, which keeps
// the caller's capture intact.
wenc_status check_sync_stream(wenc_stream_t stream, const char* what);

struct Arena {
  size_t used = 0;
  size_t take(size_t bytes) {
    size_t off = used;
    used += (bytes + 255) & ~size_t(255);
    return off;
  }
};

wenc_status check_config(const wenc_config* c) {
  if (!c) return fail(WENC_ERR_INVALID_ARG, "config is NULL");
  if (c->n_layers < 1) return fail(WENC_ERR_INVALID_ARG, "n_layers must be >= 1 (got %d)", c->n_layers);
  if (c->n_heads < 1 || c->head_dim < 1 || c->d_model < 1 || c->ffn_dim < 1 || c->seq_len < 1 || c->max_batch < 1)
    return fail(WENC_ERR_INVALID_ARG, "sizes must be positive");
  if (c->d_model != c->n_heads * c->head_dim)
    return fail(WENC_ERR_INVALID_ARG, "d_model %d != n_heads %d * head_dim %d", c->d_model, c->n_heads, c->head_dim);
  if (c->head_dim != 64) return fail(WENC_ERR_UNSUPPORTED, "head_dim %d: only 64 is implemented", c->head_dim);
  if (c->d_model % 128 != 0 || !wenc_host::layernorm_supported(c->d_model))
    return fail(WENC_ERR_UNSUPPORTED, "d_model %d: must be a multiple of 128, at most 2048", c->d_model);
  if (c->ffn_dim % 128 != 0) return fail(WENC_ERR_UNSUPPORTED, "ffn_dim %d: must be a multiple of 128", c->ffn_dim);
  if (c->seq_len > 4096) return fail(WENC_ERR_UNSUPPORTED, "seq_len %d > 4096", c->seq_len);
  if (static_cast<long long>(c->max_batch) * c->seq_len > (1LL << 28))
    return fail(WENC_ERR_UNSUPPORTED, "max_batch * seq_len too large");
  if (!(c->ln_eps >= 0.0f)) return fail(WENC_ERR_INVALID_ARG, "ln_eps must be >= 0");
  if (c->weight_dtype != WENC_DTYPE_F32 && c->weight_dtype != WENC_DTYPE_BF16)
    return fail(WENC_ERR_INVALID_ARG, "weight_dtype %d unknown", c->weight_dtype);
  if (c->precision != WENC_PREC_BF16 && c->precision != WENC_PREC_TF32)
    return fail(WENC_ERR_UNSUPPORTED, "precision %d unknown (BF16 = 0, TF32 = 1)", c->precision);
  return WENC_OK;
}

void free_handle(wenc* h) {
  if (!h) return;
  dev_free(h->weight_arena, h->weight_bytes);
  dev_free(h->work_arena, h->work_bytes);
  dev_free(h->stem_arena, h->stem_bytes);
  dev_free(h->cross_arena, h->cross_bytes);
  if (h->err_host) cudaFreeHost(h->err_host);
  delete h;
}

wenc_status check_sync_stream(wenc_stream_t stream, const char* what) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(WENC_ERR_INVALID_ARG, "%s: the stream is not usable (%s)", what, cudaGetErrorString(e));
  }
  if (cs != cudaStreamCaptureStatusNone)
    return fail(WENC_ERR_INVALID_ARG, "%s synchronises its stream and cannot run while the stream is being captured",
                what);
  return WENC_OK;
}

// One matrix into the packed arena. BF16 precision: copied (bf16 source) or rounded to bf16
// (fp32 source). TF32 precision: widened (bf16 source, exact) or rounded to TF32 (fp32 source).
cudaError_t pack_matrix(const void* src, int dtype, bool tf32, void* dst, size_t n, cudaStream_t s) {
  if (tf32) return wenc_host::launch_to_tf32(src, dtype == WENC_DTYPE_BF16, static_cast<float*>(dst), n, s);
  if (dtype == WENC_DTYPE_BF16) return cudaMemcpyAsync(dst, src, n * 2, cudaMemcpyDeviceToDevice, s);
  return wenc_host::launch_f32_to_bf16(static_cast<const float*>(src), static_cast<uint16_t*>(dst), n, s);
}

}  // namespace

namespace {

// Records each launch's kind and, when the timing hook is armed, an event after it.
struct LaunchRec {
  cudaStream_t s;
  std::vector<cudaEvent_t> ev;
  int* kinds = nullptr;
  int li = 0;
  cudaError_t e = cudaSuccess;
  void begin() {
    if (!ev.empty()) e = cudaEventRecord(ev[0], s);
  }
  void operator()(int kind, cudaError_t le) {
    if (e == cudaSuccess) e = le;
    if (kinds) kinds[li] = kind;
    ++li;
    if (!ev.empty() && e == cudaSuccess) e = cudaEventRecord(ev[li], s);
  }
};

// Common checks of the forward-type entry points; takes the armed timing hook (which clears it).
wenc_status begin_call(wenc* h, const void* in, const void* out, int B, int n_launch, cudaStream_t s, LaunchRec* rec) {
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  if (!in || !out) return fail(WENC_ERR_INVALID_ARG, "input/output buffer is NULL");
  if (!aligned16(in) || !aligned16(out)) return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (B < 1 || B > h->cfg.max_batch)
    return fail(WENC_ERR_INVALID_ARG, "B = %d outside 1..max_batch %d", B, h->cfg.max_batch);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != h->device) return fail(WENC_ERR_INVALID_ARG, "current device %d is not the handle's device %d", dev, h->device);
  if (*reinterpret_cast<volatile uint32_t*>(h->err_host) != 0)
    return fail(WENC_ERR_DEVICE_TIMEOUT, "an earlier launch recorded device error word 0x%x",
                *reinterpret_cast<volatile uint32_t*>(h->err_host));
  rec->s = s;
  rec->ev.swap(h->events);
  h->events.clear();
  rec->kinds = h->kinds;
  h->kinds = nullptr;
  if (!rec->ev.empty() && static_cast<int>(rec->ev.size()) < n_launch + 1)
    return fail(WENC_ERR_INVALID_ARG, "launch events: need %d, got %zu", n_launch + 1, rec->ev.size());
  rec->begin();
  return WENC_OK;
}

// The stem's four launches: mel [B, 2T, n_mels] -> x [B, T, d] (fp32).
void enqueue_stem(wenc* h, const float* mel, float* x, int B, LaunchRec& rec) {
  const wenc_config& c = h->cfg;
  const int d = c.d_model, T = c.seq_len;
  rec(9, wenc_host::launch_unfold3(mel, true, h->a1, h->tf32, B, 2 * T, h->n_mels, 1, h->kp1, rec.s));
  rec(10, wenc_host::launch_gemm(h->tm_a1, h->tm_wc1, B * 2 * T, d, h->kp1, h->bn_stem, WENC_EPI_BIAS_GELU_BF16,
                                 h->cb1, nullptr, h->h1, h->err_dev, h->num_sms, rec.s, h->tf32, 0,
                                 wenc_host::GemmExtra(), &h->tm_wc1_h));
  rec(9, wenc_host::launch_unfold3(h->h1, h->tf32, h->a2, h->tf32, B, 2 * T, d, 2, 3 * d, rec.s));
  rec(11, wenc_host::launch_gemm(h->tm_a2, h->tm_wc2, B * T, d, 3 * d, h->bn_stem, wenc_host::kEpiGeluTable, h->cb2,
                                 h->pos, x, h->err_dev, h->num_sms, rec.s, h->tf32, T,
                                 wenc_host::GemmExtra(), &h->tm_wc2_h));
}

// The blocks first .. first+count-1 and, if final_ln, the final LayerNorm: in -> out.
// Optional NVTX ranges (WENC_NVTX=1 in the environment): one range per block around its launches,
// named "wenc block <l>", so that a profiler can select a block's kernels (for example with ncu's
// --nvtx --nvtx-include "wenc block 5/"). Off by default: then no NVTX call is made.
bool nvtx_enabled() {
  static const bool on = [] {
    const char* v = getenv("WENC_NVTX");
    return v && v[0] == '1';
  }();
  return on;
}

struct NvtxRange {
  bool on;
  explicit NvtxRange(int layer) : on(nvtx_enabled()) {
    if (!on) return;
    char name[32];
    snprintf(name, sizeof(name), "wenc block %d", layer);
    nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
};

void enqueue_blocks(wenc* h, const float* in, float* out, int B, int first, int count, bool final_ln, LaunchRec& rec) {
  const wenc_config& c = h->cfg;
  const cudaStream_t s = rec.s;
  const int d = c.d_model, f = c.ffn_dim, T = c.seq_len, H = c.n_heads;
  const int M = B * T;
  const float* src = in;  // the residual stream entering the next block
  if (!h->tf32 && count > 0)  // statistics and bf16 copy of the first block's input
    rec(14, wenc_host::launch_row_stats(in, static_cast<uint16_t*>(h->xn), h->stats, M, d, h->seg_w, s));
  for (int l = first; l < first + count && rec.e == cudaSuccess; ++l) {
    const NvtxRange range(l);
    const wenc::Layer& P = h->layers[l];
    const bool last = (l == first + count - 1);
    float* dst_final = (last && !final_ln) ? out : h->x;
    if (h->tf32) {
      // TF32: every GEMM operand is fp32 rounded to TF32 by its producer.
      rec(0, wenc_host::launch_layernorm(src, P.ln1_w, P.ln1_b, h->xn, M, d, c.ln_eps, 2, s));
      rec(1, wenc_host::launch_gemm(h->tm_xn, P.tm_wqkv, M, 3 * d, d, h->bn_qkv, WENC_EPI_BIAS_BF16, P.bqkv, nullptr,
                                    h->qkv, h->err_dev, h->num_sms, s, true, 0, {}, &P.tm_wqkv_h));
      rec(2, wenc_host::launch_attention_tf32(h->tm_q, h->tm_kv, h->tm_kv, 0, d, 2 * d, static_cast<float*>(h->o), d,
                                              B, T, H, h->err_dev, s));
      rec(3, wenc_host::launch_gemm(h->tm_o, P.tm_wo, M, d, d, h->bn_o, WENC_EPI_BIAS_RESID_F32, P.bo, src, h->x,
                                    h->err_dev, h->num_sms, s, true, 0, {}, &P.tm_wo_h));
      rec(0, wenc_host::launch_layernorm(h->x, P.ln2_w, P.ln2_b, h->xn, M, d, c.ln_eps, 2, s));
      rec(4, wenc_host::launch_gemm(h->tm_xn, P.tm_w1, M, f, d, h->bn_1, WENC_EPI_BIAS_GELU_BF16, P.b1, nullptr, h->u,
                                    h->err_dev, h->num_sms, s, true, 0, {}, &P.tm_w1_h));
      rec(5, wenc_host::launch_gemm(h->tm_u, P.tm_w2, M, d, f, h->bn_2, WENC_EPI_BIAS_RESID_F32, P.b2, h->x, dst_final,
                                    h->err_dev, h->num_sms, s, true, 0, {}, &P.tm_w2_h));
      src = h->x;
      continue;
    }
    // BF16: LN1 is folded into the QKV GEMM, which reads the raw residual stream (its bf16 copy
    // in xn) and the row statistics written by the previous block's fc2 epilogue (or, for the
    // call's first block, by the row-statistics kernel). LN2 stays a kernel of its own: folding
    // it too would move more work into the out-projection and fc1 epilogues than it saves.
    uint16_t* o16 = static_cast<uint16_t*>(h->o);
    uint16_t* xn16 = static_cast<uint16_t*>(h->xn);
    wenc_host::GemmExtra ln1, wr;
    ln1.colsum = P.cs_qkv;
    ln1.stats = h->stats;
    ln1.eps = c.ln_eps;
    ln1.seg_w = wr.seg_w = h->seg_w;
    wr.copy = xn16;
    wr.stats_out = h->stats;
    rec(1, wenc_host::launch_gemm(h->tm_xn, P.tm_wqkv, M, 3 * d, d, h->bn_qkv, wenc_host::kEpiLnBias, P.bqkv, nullptr,
                                  h->qkv, h->err_dev, h->num_sms, s, false, 0, ln1, &P.tm_wqkv_h));
    rec(2, wenc_host::launch_attention_main(h->tm_q, h->tm_kv, h->tm_kv, 0, d, 2 * d, o16, d, B, T, H, h->err_dev, s,
                                            h->attn_splits, h->part_o, h->part_ml));
    if (wenc_host::attention_launches(T, h->attn_splits) == 2)
      rec(8, wenc_host::launch_attention_combine(h->part_o, h->part_ml, o16, d, B, T, H, h->attn_splits, s));
    rec(3, wenc_host::launch_gemm(h->tm_o, P.tm_wo, M, d, d, h->bn_o, WENC_EPI_BIAS_RESID_F32, P.bo, src, h->x,
                                  h->err_dev, h->num_sms, s, false, 0, {}, &P.tm_wo_h));
    rec(0, wenc_host::launch_layernorm(h->x, P.ln2_w, P.ln2_b, h->xn, M, d, c.ln_eps, 1, s));
    rec(4, wenc_host::launch_gemm(h->tm_xn, P.tm_w1, M, f, d, h->bn_1, WENC_EPI_BIAS_GELU_BF16, P.b1, nullptr, h->u,
                                  h->err_dev, h->num_sms, s, false, 0, {}, &P.tm_w1_h));
    if (last)  // the call's output: the final LayerNorm (its own kernel) or the caller reads it
      rec(5, wenc_host::launch_gemm(h->tm_u, P.tm_w2, M, d, f, h->bn_2, WENC_EPI_BIAS_RESID_F32, P.b2, h->x, dst_final,
                                    h->err_dev, h->num_sms, s, false, 0, {}, &P.tm_w2_h));
    else
      rec(5, wenc_host::launch_gemm(h->tm_u, P.tm_w2, M, d, f, h->bn_2, wenc_host::kEpiResidStats, P.b2, h->x, dst_final,
                                    h->err_dev, h->num_sms, s, false, 0, wr, &P.tm_w2_h));
    src = h->x;
  }
  if (rec.e == cudaSuccess) {
    if (final_ln) {
      rec(6, wenc_host::launch_layernorm(src, h->lnf_w, h->lnf_b, out, M, d, c.ln_eps, 0, s));
    } else if (count == 0) {
      rec(7, in == out ? cudaSuccess : cudaMemcpyAsync(out, in, size_t(M) * d * 4, cudaMemcpyDeviceToDevice, s));
    }
  }
}

}  // namespace

// Helpers shared with the other entry-point files (status message, error word, device checks).
wenc_status wenc_internal_fail(wenc_status s, const char* msg) { return fail(s, "%s", msg); }
void wenc_internal_clear_error() { g_last_error.clear(); }
uint32_t* wenc_internal_error_word(std::string* why) { return global_error_word(why); }
bool wenc_internal_is_sm103(std::string* why) { return device_is_sm103(why); }
int wenc_internal_sm_count() { return sm_count(); }

extern "C" {

const char* wenc_last_error(void) { return g_last_error.c_str(); }

void wenc_set_device_alloc_limit(size_t bytes) { g_dev_limit.store(bytes); }

size_t wenc_device_bytes_held(void) { return g_dev_held.load(); }

const char* wenc_version(void) { return "wenc 0.1 sm_103a"; }

wenc_status wenc_create(const wenc_config* cfg, const wenc_layer_weights* layers, const float* lnf_w,
                        const float* lnf_b, wenc_stream_t stream_, wenc** out) {
  g_last_error.clear();
  if (!out) return fail(WENC_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  wenc_status st = check_config(cfg);
  if (st != WENC_OK) return st;
  if (!layers) return fail(WENC_ERR_INVALID_ARG, "layers is NULL");
  std::string why;
  if (!device_is_sm103(&why)) return fail(WENC_ERR_UNSUPPORTED, "%s", why.c_str());
  st = check_sync_stream(stream_, "wenc_create");
  if (st != WENC_OK) return st;
  const int L = cfg->n_layers, d = cfg->d_model, f = cfg->ffn_dim;
  for (int l = 0; l < L; ++l) {
    const wenc_layer_weights& w = layers[l];
    const void* req[] = {w.ln1_w, w.ln1_b, w.wq, w.bq, w.wk, w.wv, w.bv, w.wo, w.bo,
                         w.ln2_w, w.ln2_b, w.w1, w.b1, w.w2, w.b2};
    for (const void* p : req) {
      if (!p) return fail(WENC_ERR_INVALID_ARG, "layer %d: a required weight pointer is NULL", l);
      if (!is_device_accessible(p)) return fail(WENC_ERR_INVALID_ARG, "layer %d: a weight pointer is not device memory", l);
    }
    if (w.bk) return fail(WENC_ERR_INVALID_ARG, "layer %d: bk must be NULL (the K projection has no bias)", l);
  }
  if (cfg->final_ln && (!lnf_w || !lnf_b)) return fail(WENC_ERR_INVALID_ARG, "final_ln set but lnf_w/lnf_b NULL");
  if (cfg->final_ln && (!is_device_accessible(lnf_w) || !is_device_accessible(lnf_b)))
    return fail(WENC_ERR_INVALID_ARG, "lnf_w/lnf_b are not device memory");

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_);
  wenc* h = new wenc();
  h->cfg = *cfg;
  cudaGetDevice(&h->device);
  h->num_sms = sm_count();
  h->tf32 = cfg->precision == WENC_PREC_TF32;
  h->esz = h->tf32 ? 4 : 2;
  const size_t es = h->esz;
  h->bn_qkv = wenc_host::gemm_pick_bn(3 * d);
  h->bn_o = wenc_host::gemm_pick_bn(d);
  h->bn_1 = wenc_host::gemm_pick_bn(f);
  h->bn_2 = wenc_host::gemm_pick_bn(d);

  // ---- weights arena
  Arena wa;
  struct Off { size_t wqkv, wo, w1, w2, ln1_w, ln1_b, bqkv, bo, ln2_w, ln2_b, b1, b2, cs_qkv; };
  std::vector<Off> offs(L);
  for (int l = 0; l < L; ++l) {
    Off& o = offs[l];
    o.wqkv = wa.take(size_t(3) * d * d * es);
    o.wo = wa.take(size_t(d) * d * es);
    o.w1 = wa.take(size_t(f) * d * es);
    o.w2 = wa.take(size_t(d) * f * es);
    o.ln1_w = wa.take(d * 4); o.ln1_b = wa.take(d * 4);
    o.bqkv = wa.take(3 * d * 4); o.bo = wa.take(d * 4);
    o.ln2_w = wa.take(d * 4); o.ln2_b = wa.take(d * 4);
    o.b1 = wa.take(f * 4); o.b2 = wa.take(d * 4);
    if (!h->tf32) o.cs_qkv = wa.take(3 * d * 4);
  }
  const size_t off_lnf_w = wa.take(d * 4), off_lnf_b = wa.take(d * 4);
  cudaError_t e = dev_alloc(&h->weight_arena, wa.used);
  if (e == cudaSuccess) h->weight_bytes = wa.used;
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return fail(WENC_ERR_OOM, "weights: cudaMalloc(%zu) failed", wa.used);
  }
  uint8_t* wb = static_cast<uint8_t*>(h->weight_arena);

  // ---- workspace arena
  const size_t rows = size_t(cfg->max_batch) * cfg->seq_len;
  Arena ka;
  const size_t off_x = ka.take(rows * d * 4), off_xn = ka.take(rows * d * es), off_qkv = ka.take(rows * 3 * d * es),
               off_o = ka.take(rows * d * es), off_u = ka.take(rows * f * es);
  // BF16: the per-row segment statistics the LayerNorm-folded GEMMs read (segments of bn / 2
  // columns, bn the tile width of the GEMMs that write the residual stream)
  h->seg_w = wenc_host::gemm_pick_bn(d) / 2;
  const size_t off_stats = h->tf32 ? 0 : ka.take(rows * (d / h->seg_w) * sizeof(float2));
  // Small batches leave most SMs idle in attention: split the keys among more CTAs then (the
  // bf16 kernel only).
  h->attn_splits =
      h->tf32 ? 1 : wenc_host::attention_pick_splits(cfg->max_batch, cfg->seq_len, cfg->n_heads, h->num_sms);
  const size_t part_rows = static_cast<size_t>(h->attn_splits) * cfg->max_batch * cfg->n_heads * cfg->seq_len;
  const size_t off_po = h->attn_splits > 1 ? ka.take(part_rows * wenc_host::kAttnHD * sizeof(float)) : 0;
  const size_t off_pml = h->attn_splits > 1 ? ka.take(part_rows * sizeof(float2)) : 0;
  e = dev_alloc(&h->work_arena, ka.used);
  if (e == cudaSuccess) h->work_bytes = ka.used;
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return fail(WENC_ERR_OOM, "workspace: cudaMalloc(%zu) failed", ka.used);
  }
  uint8_t* kb = static_cast<uint8_t*>(h->work_arena);
  h->x = reinterpret_cast<float*>(kb + off_x);
  h->xn = kb + off_xn;
  h->qkv = kb + off_qkv;
  h->o = kb + off_o;
  h->u = kb + off_u;
  if (!h->tf32) h->stats = reinterpret_cast<float2*>(kb + off_stats);
  if (h->attn_splits > 1) {
    h->part_o = reinterpret_cast<float*>(kb + off_po);
    h->part_ml = reinterpret_cast<float2*>(kb + off_pml);
  }

  e = cudaHostAlloc(reinterpret_cast<void**>(&h->err_host), sizeof(uint32_t), cudaHostAllocMapped);
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return fail(WENC_ERR_OOM, "error word: cudaHostAlloc failed");
  }
  *h->err_host = 0;
  cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->err_dev), h->err_host, 0);

  // ---- pack weights
  h->layers.resize(L);
  for (int l = 0; l < L && e == cudaSuccess; ++l) {
    const wenc_layer_weights& w = layers[l];
    const Off& o = offs[l];
    wenc::Layer& P = h->layers[l];
    P.wqkv = wb + o.wqkv;
    P.wo = wb + o.wo;
    P.w1 = wb + o.w1;
    P.w2 = wb + o.w2;
    P.ln1_w = reinterpret_cast<float*>(wb + o.ln1_w);
    P.ln1_b = reinterpret_cast<float*>(wb + o.ln1_b);
    P.bqkv = reinterpret_cast<float*>(wb + o.bqkv);
    P.bo = reinterpret_cast<float*>(wb + o.bo);
    P.ln2_w = reinterpret_cast<float*>(wb + o.ln2_w);
    P.ln2_b = reinterpret_cast<float*>(wb + o.ln2_b);
    P.b1 = reinterpret_cast<float*>(wb + o.b1);
    P.b2 = reinterpret_cast<float*>(wb + o.b2);
    const size_t dd = size_t(d) * d;
    uint8_t* qkv_w = static_cast<uint8_t*>(P.wqkv);
    const int wdt = cfg->weight_dtype;
    auto cp = [&](float* dst, const float* src, size_t n) {
      if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, n * 4, cudaMemcpyDeviceToDevice, s);
    };
    if (h->tf32) {
      if (e == cudaSuccess) e = pack_matrix(w.wq, wdt, h->tf32, qkv_w, dd, s);
      if (e == cudaSuccess) e = pack_matrix(w.wk, wdt, h->tf32, qkv_w + dd * es, dd, s);
      if (e == cudaSuccess) e = pack_matrix(w.wv, wdt, h->tf32, qkv_w + 2 * dd * es, dd, s);
      if (e == cudaSuccess) e = pack_matrix(w.w1, wdt, h->tf32, P.w1, size_t(f) * d, s);
      cp(P.bqkv, w.bq, d);
      if (e == cudaSuccess) e = cudaMemsetAsync(P.bqkv + d, 0, size_t(d) * 4, s);  // K has no bias
      cp(P.bqkv + 2 * d, w.bv, d);
      cp(P.b1, w.b1, f);
    } else {
      // LN1 folded into Q, K, V (K's own bias is absent; its folded bias is Wk ln1_b):
      // W' = bf16(W diag(ln1_w)), the row sums of W', bias' = W ln1_b + bias
      P.cs_qkv = reinterpret_cast<float*>(wb + o.cs_qkv);
      const bool wbf = wdt == WENC_DTYPE_BF16;
      uint16_t* q16 = reinterpret_cast<uint16_t*>(qkv_w);
      const void* srcs[3] = {w.wq, w.wk, w.wv};
      const float* bsrc[3] = {w.bq, nullptr, w.bv};
      for (int i = 0; i < 3 && e == cudaSuccess; ++i)
        e = wenc_host::launch_fold_ln(srcs[i], wbf, w.ln1_w, w.ln1_b, bsrc[i], q16 + i * dd, P.cs_qkv + i * d,
                                      P.bqkv + i * d, d, d, s);
      if (e == cudaSuccess) e = pack_matrix(w.w1, wdt, false, P.w1, size_t(f) * d, s);
      cp(P.b1, w.b1, f);
    }
    if (e == cudaSuccess) e = pack_matrix(w.wo, wdt, h->tf32, P.wo, dd, s);
    if (e == cudaSuccess) e = pack_matrix(w.w2, wdt, h->tf32, P.w2, size_t(d) * f, s);
    cp(P.ln1_w, w.ln1_w, d); cp(P.ln1_b, w.ln1_b, d);
    cp(P.bo, w.bo, d);
    cp(P.ln2_w, w.ln2_w, d); cp(P.ln2_b, w.ln2_b, d);
    cp(P.b2, w.b2, d);
  }
  if (cfg->final_ln && e == cudaSuccess) {
    h->lnf_w = reinterpret_cast<float*>(wb + off_lnf_w);
    h->lnf_b = reinterpret_cast<float*>(wb + off_lnf_b);
    e = cudaMemcpyAsync(h->lnf_w, lnf_w, d * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->lnf_b, lnf_b, d * 4, cudaMemcpyDeviceToDevice, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    free_handle(h);
    return cuda_fail(e, "packing weights");
  }

  // ---- tensor maps (all over library-owned buffers; built once). A stage row is 128 bytes:
  // 64 bf16 or 32 fp32 elements.
  bool ok = true;
  const uint32_t kbox = h->tf32 ? 32 : 64;
  auto map2 = [&](CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    ok = ok && (h->tf32 ? wenc_host::make_tmap_2d_f32(m, base, inner, outer, inner * 4, kbox, box_outer, &why)
                        : wenc_host::make_tmap_2d_bf16(m, base, inner, outer, inner * 2, kbox, box_outer, &why));
  };
  for (int l = 0; l < L && ok; ++l) {
    wenc::Layer& P = h->layers[l];
    map2(&P.tm_wqkv, P.wqkv, d, 3 * d, h->bn_qkv);
    map2(&P.tm_wo, P.wo, d, d, h->bn_o);
    map2(&P.tm_w1, P.w1, d, f, h->bn_1);
    map2(&P.tm_w2, P.w2, f, d, h->bn_2);
    map2(&P.tm_wqkv_h, P.wqkv, d, 3 * d, h->bn_qkv / 2);
    map2(&P.tm_wo_h, P.wo, d, d, h->bn_o / 2);
    map2(&P.tm_w1_h, P.w1, d, f, h->bn_1 / 2);
    map2(&P.tm_w2_h, P.w2, f, d, h->bn_2 / 2);
  }
  map2(&h->tm_xn, h->xn, d, rows, wenc_host::kGemmBM);
  map2(&h->tm_o, h->o, d, rows, wenc_host::kGemmBM);
  map2(&h->tm_u, h->u, f, rows, wenc_host::kGemmBM);
  const size_t qkv_row = size_t(3) * d * es;
  if (h->tf32) {
    ok = ok && wenc_host::make_tmap_3d_f32(&h->tm_q, h->qkv, 3 * d, cfg->seq_len, cfg->max_batch, qkv_row,
                                           qkv_row * cfg->seq_len, 32, wenc_host::kAttnTf32BQ, &why);
    ok = ok && wenc_host::make_tmap_3d_f32(&h->tm_kv, h->qkv, 3 * d, cfg->seq_len, cfg->max_batch, qkv_row,
                                           qkv_row * cfg->seq_len, 32, wenc_host::kAttnTf32BKV, &why);
  } else {
    ok = ok && wenc_host::make_tmap_3d_bf16(&h->tm_q, h->qkv, 3 * d, cfg->seq_len, cfg->max_batch, qkv_row,
                                            qkv_row * cfg->seq_len, 64, wenc_host::kAttnBQ, &why);
    ok = ok && wenc_host::make_tmap_3d_bf16(&h->tm_kv, h->qkv, 3 * d, cfg->seq_len, cfg->max_batch, qkv_row,
                                            qkv_row * cfg->seq_len, 64, wenc_host::kAttnBKV, &why);
  }
  if (!ok) {
    free_handle(h);
    return fail(WENC_ERR_CUDA, "%s", why.c_str());
  }
  *out = h;
  return WENC_OK;
}

int wenc_forward_launches(const wenc* h, int first, int count, int apply_final_ln) {
  if (!h || first < 0 || count < 0 || first + count > h->cfg.n_layers) return -1;
  const bool final_ln = apply_final_ln && h->cfg.final_ln;
  const int attn = h->tf32 ? 1 : wenc_host::attention_launches(h->cfg.seq_len, h->attn_splits);
  // TF32: LN1, QKV, attention, out-proj, LN2, fc1, fc2 per block. BF16: LN1 is folded into the
  // QKV GEMM, plus one row-statistics launch for the first block's input.
  int n = h->tf32 ? (6 + attn) * count : (5 + attn) * count + (count > 0 ? 1 : 0);
  if (final_ln) n += 1;
  else if (count == 0) n += 1;  // the copy in -> out
  return n;
}

wenc_status wenc_set_launch_events(wenc* h, void* const* events, int n_events, int* kinds) {
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  h->events.clear();
  h->kinds = kinds;
  if (events) {
    if (n_events < 1) return fail(WENC_ERR_INVALID_ARG, "n_events < 1");
    for (int i = 0; i < n_events; ++i) h->events.push_back(static_cast<cudaEvent_t>(events[i]));
  }
  return WENC_OK;
}

wenc_status wenc_forward_layers(wenc* h, const float* in, float* out, int B, int first, int count, int apply_final_ln,
                                wenc_stream_t stream_) {
  g_last_error.clear();
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  const wenc_config& c = h->cfg;
  if (first < 0 || count < 0 || first + count > c.n_layers)
    return fail(WENC_ERR_INVALID_ARG, "layers %d..%d outside 0..%d", first, first + count - 1, c.n_layers - 1);
  LaunchRec rec;
  wenc_status st = begin_call(h, in, out, B, wenc_forward_launches(h, first, count, apply_final_ln),
                              reinterpret_cast<cudaStream_t>(stream_), &rec);
  if (st != WENC_OK) return st;
  enqueue_blocks(h, in, out, B, first, count, apply_final_ln && c.final_ln, rec);
  if (rec.e != cudaSuccess) return cuda_fail(rec.e, "forward launch");
  return WENC_OK;
}

wenc_status wenc_forward(wenc* h, const float* in, float* out, int B, wenc_stream_t stream) {
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  return wenc_forward_layers(h, in, out, B, 0, h->cfg.n_layers, 1, stream);
}

wenc_status wenc_set_stem(wenc* h, const wenc_stem_weights* w, wenc_stream_t stream_) {
  g_last_error.clear();
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  if (!w) return fail(WENC_ERR_INVALID_ARG, "stem weights are NULL");
  const void* req[] = {w->conv1_w, w->conv1_b, w->conv2_w, w->conv2_b, w->positions};
  for (const void* p : req) {
    if (!p) return fail(WENC_ERR_INVALID_ARG, "a stem weight pointer is NULL");
    if (!is_device_accessible(p)) return fail(WENC_ERR_INVALID_ARG, "a stem weight pointer is not device memory");
  }
  if (w->n_mels < 8 || w->n_mels > 1024 || w->n_mels % 8 != 0)
    return fail(WENC_ERR_INVALID_ARG, "n_mels %d: a multiple of 8 in 8..1024", w->n_mels);
  const wenc_status sst = check_sync_stream(stream_, "wenc_set_stem");
  if (sst != WENC_OK) return sst;
  const wenc_config& c = h->cfg;
  const int d = c.d_model, T = c.seq_len, nm = w->n_mels;
  const size_t es = h->esz;
  const int kp1 = (3 * nm + 63) / 64 * 64;  // conv1's K, padded to whole 64-element stages
  const size_t rows1 = size_t(c.max_batch) * 2 * T, rows2 = size_t(c.max_batch) * T;
  Arena ar;
  const size_t o_wc1 = ar.take(size_t(d) * kp1 * es), o_wc2 = ar.take(size_t(d) * 3 * d * es);
  const size_t o_cb1 = ar.take(size_t(d) * 4), o_cb2 = ar.take(size_t(d) * 4), o_pos = ar.take(size_t(T) * d * 4);
  const size_t o_a1 = ar.take(rows1 * kp1 * es), o_h1 = ar.take(rows1 * d * es), o_a2 = ar.take(rows2 * 3 * d * es);
  if (h->stem_arena) {
    cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_));
    dev_free(h->stem_arena, h->stem_bytes);
  }
  h->has_stem = false;
  cudaError_t e = dev_alloc(&h->stem_arena, ar.used);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(WENC_ERR_OOM, "stem: cudaMalloc(%zu) failed", ar.used);
  }
  h->stem_bytes = ar.used;
  uint8_t* base = static_cast<uint8_t*>(h->stem_arena);
  h->n_mels = nm;
  h->kp1 = kp1;
  h->bn_stem = wenc_host::gemm_pick_bn(d);
  h->wc1 = base + o_wc1;
  h->wc2 = base + o_wc2;
  h->cb1 = reinterpret_cast<float*>(base + o_cb1);
  h->cb2 = reinterpret_cast<float*>(base + o_cb2);
  h->pos = reinterpret_cast<float*>(base + o_pos);
  h->a1 = base + o_a1;
  h->h1 = base + o_h1;
  h->a2 = base + o_a2;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_);
  const bool wbf16 = c.weight_dtype == WENC_DTYPE_BF16;
  e = wenc_host::launch_conv_weight(w->conv1_w, wbf16, h->wc1, h->tf32, d, nm, kp1, s);
  if (e == cudaSuccess) e = wenc_host::launch_conv_weight(w->conv2_w, wbf16, h->wc2, h->tf32, d, d, 3 * d, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->cb1, w->conv1_b, size_t(d) * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->cb2, w->conv2_b, size_t(d) * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->pos, w->positions, size_t(T) * d * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "packing the stem");
  std::string why;
  const uint32_t kbox = h->tf32 ? 32 : 64;
  bool ok = true;
  auto map2 = [&](CUtensorMap* m, const void* p, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    ok = ok && (h->tf32 ? wenc_host::make_tmap_2d_f32(m, p, inner, outer, inner * 4, kbox, box_outer, &why)
                        : wenc_host::make_tmap_2d_bf16(m, p, inner, outer, inner * 2, kbox, box_outer, &why));
  };
  map2(&h->tm_a1, h->a1, kp1, rows1, wenc_host::kGemmBM);
  map2(&h->tm_wc1, h->wc1, kp1, d, h->bn_stem);
  map2(&h->tm_a2, h->a2, 3 * d, rows2, wenc_host::kGemmBM);
  map2(&h->tm_wc2, h->wc2, 3 * d, d, h->bn_stem);
  map2(&h->tm_wc1_h, h->wc1, kp1, d, h->bn_stem / 2);
  map2(&h->tm_wc2_h, h->wc2, 3 * d, d, h->bn_stem / 2);
  if (!ok) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  h->has_stem = true;
  return WENC_OK;
}

int wenc_encode_launches(const wenc* h) {
  if (!h || !h->has_stem) return -1;
  return 4 + wenc_forward_launches(h, 0, h->cfg.n_layers, 1);
}

wenc_status wenc_stem(wenc* h, const float* mel, float* out, int B, wenc_stream_t stream_) {
  g_last_error.clear();
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  if (!h->has_stem) return fail(WENC_ERR_INVALID_ARG, "no stem: call wenc_set_stem first");
  LaunchRec rec;
  wenc_status st = begin_call(h, mel, out, B, 4, reinterpret_cast<cudaStream_t>(stream_), &rec);
  if (st != WENC_OK) return st;
  enqueue_stem(h, mel, out, B, rec);
  if (rec.e != cudaSuccess) return cuda_fail(rec.e, "stem launch");
  return WENC_OK;
}

wenc_status wenc_encode(wenc* h, const float* mel, float* out, int B, wenc_stream_t stream_) {
  g_last_error.clear();
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  if (!h->has_stem) return fail(WENC_ERR_INVALID_ARG, "no stem: call wenc_set_stem first");
  LaunchRec rec;
  wenc_status st = begin_call(h, mel, out, B, wenc_encode_launches(h), reinterpret_cast<cudaStream_t>(stream_), &rec);
  if (st != WENC_OK) return st;
  enqueue_stem(h, mel, h->x, B, rec);  // the stem writes the residual stream the blocks start from
  if (rec.e == cudaSuccess) enqueue_blocks(h, h->x, out, B, 0, h->cfg.n_layers, h->cfg.final_ln != 0, rec);
  if (rec.e != cudaSuccess) return cuda_fail(rec.e, "encode launch");
  return WENC_OK;
}

wenc_status wenc_set_cross_kv(wenc* h, int n_dec, const void* const* wk, const void* const* wv, const float* const* bv,
                              wenc_stream_t stream_) {
  g_last_error.clear();
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  if (n_dec < 1) return fail(WENC_ERR_INVALID_ARG, "n_dec_layers must be >= 1 (got %d)", n_dec);
  if (!wk || !wv || !bv) return fail(WENC_ERR_INVALID_ARG, "wk/wv/bv arrays are NULL");
  for (int l = 0; l < n_dec; ++l) {
    const void* req[] = {wk[l], wv[l], bv[l]};
    for (const void* p : req) {
      if (!p) return fail(WENC_ERR_INVALID_ARG, "decoder layer %d: a cross K/V pointer is NULL", l);
      if (!is_device_accessible(p)) return fail(WENC_ERR_INVALID_ARG, "decoder layer %d: not device memory", l);
    }
  }
  const wenc_status sst = check_sync_stream(stream_, "wenc_set_cross_kv");
  if (sst != WENC_OK) return sst;
  const wenc_config& c = h->cfg;
  const int d = c.d_model;
  const size_t es = h->esz, n_out = size_t(2) * n_dec * d;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_);
  if (h->cross_arena) {
    cudaStreamSynchronize(s);
    dev_free(h->cross_arena, h->cross_bytes);
  }
  h->n_dec = 0;
  Arena ar;
  const size_t o_w = ar.take(n_out * d * es), o_b = ar.take(n_out * 4);
  cudaError_t e = dev_alloc(&h->cross_arena, ar.used);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(WENC_ERR_OOM, "cross K/V: cudaMalloc(%zu) failed", ar.used);
  }
  h->cross_bytes = ar.used;
  uint8_t* base = static_cast<uint8_t*>(h->cross_arena);
  h->wx = base + o_w;
  h->bx = reinterpret_cast<float*>(base + o_b);
  const size_t dd = size_t(d) * d;
  for (int l = 0; l < n_dec && e == cudaSuccess; ++l) {
    uint8_t* wl = static_cast<uint8_t*>(h->wx) + size_t(2) * l * dd * es;
    e = pack_matrix(wk[l], c.weight_dtype, h->tf32, wl, dd, s);
    if (e == cudaSuccess) e = pack_matrix(wv[l], c.weight_dtype, h->tf32, wl + dd * es, dd, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->bx + size_t(2) * l * d, 0, size_t(d) * 4, s);  // K: no bias
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->bx + size_t(2 * l + 1) * d, bv[l], size_t(d) * 4, cudaMemcpyDeviceToDevice, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "packing the cross K/V weights");
  h->bn_cross = wenc_host::gemm_pick_bn(static_cast<int>(n_out));
  std::string why;
  const bool ok =
      h->tf32 ? (wenc_host::make_tmap_2d_f32(&h->tm_wx, h->wx, d, n_out, size_t(d) * 4, 32, h->bn_cross, &why) &&
                 wenc_host::make_tmap_2d_f32(&h->tm_wx_h, h->wx, d, n_out, size_t(d) * 4, 32, h->bn_cross / 2, &why))
              : (wenc_host::make_tmap_2d_bf16(&h->tm_wx, h->wx, d, n_out, size_t(d) * 2, 64, h->bn_cross, &why) &&
                 wenc_host::make_tmap_2d_bf16(&h->tm_wx_h, h->wx, d, n_out, size_t(d) * 2, 64, h->bn_cross / 2, &why));
  if (!ok) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  h->n_dec = n_dec;
  return WENC_OK;
}

wenc_status wenc_cross_kv(wenc* h, const float* enc_out, void* kv_out, int B, wenc_stream_t stream_) {
  g_last_error.clear();
  if (!h) return fail(WENC_ERR_INVALID_ARG, "handle is NULL");
  if (h->n_dec < 1) return fail(WENC_ERR_INVALID_ARG, "no cross K/V weights: call wenc_set_cross_kv first");
  LaunchRec rec;
  wenc_status st = begin_call(h, enc_out, kv_out, B, 2, reinterpret_cast<cudaStream_t>(stream_), &rec);
  if (st != WENC_OK) return st;
  const int d = h->cfg.d_model, M = B * h->cfg.seq_len;
  const size_t n = size_t(M) * d;
  // the encoder output in the operand format, in the LayerNorm-output workspace
  rec(12, h->tf32 ? wenc_host::launch_to_tf32(enc_out, false, static_cast<float*>(h->xn), n, rec.s)
                  : wenc_host::launch_f32_to_bf16(enc_out, static_cast<uint16_t*>(h->xn), n, rec.s));
  rec(13, wenc_host::launch_gemm(h->tm_xn, h->tm_wx, M, 2 * h->n_dec * d, d, h->bn_cross, wenc_host::kEpiBiasPlanes,
                                 h->bx, nullptr, kv_out, h->err_dev, h->num_sms, rec.s, h->tf32, d,
                                 wenc_host::GemmExtra(), &h->tm_wx_h));
  if (rec.e != cudaSuccess) return cuda_fail(rec.e, "cross K/V launch");
  return WENC_OK;
}

wenc_status wenc_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* out, int B, int T, int H,
                           int hd, wenc_stream_t stream) {
  g_last_error.clear();
  if (!q || !k || !v || !out) return fail(WENC_ERR_INVALID_ARG, "q/k/v/out is NULL");
  if (B < 1 || T < 1 || H < 1) return fail(WENC_ERR_INVALID_ARG, "B, T, H must be >= 1");
  if (hd != 64) return fail(WENC_ERR_UNSUPPORTED, "head_dim %d: only 64 is implemented", hd);
  if (T > (1 << 20)) return fail(WENC_ERR_UNSUPPORTED, "T %d too large", T);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  std::string why;
  if (!device_is_sm103(&why)) return fail(WENC_ERR_UNSUPPORTED, "%s", why.c_str());
  uint32_t* err = global_error_word(&why);
  if (!err) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  const uint64_t row = uint64_t(H) * 64;
  CUtensorMap tq, tk, tv;
  bool ok = wenc_host::make_tmap_3d_bf16(&tq, q, row, T, B, row * 2, row * 2 * T, 64, wenc_host::kAttnBQ, &why) &&
            wenc_host::make_tmap_3d_bf16(&tk, k, row, T, B, row * 2, row * 2 * T, 64, wenc_host::kAttnBKV, &why) &&
            wenc_host::make_tmap_3d_bf16(&tv, v, row, T, B, row * 2, row * 2 * T, 64, wenc_host::kAttnBKV, &why);
  if (!ok) return fail(WENC_ERR_INVALID_ARG, "%s", why.c_str());
  cudaError_t e = wenc_host::launch_attention(tq, tk, tv, 0, 0, 0, out, static_cast<int>(row), B, T, H, err,
                                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return WENC_OK;
}

wenc_status wenc_layernorm(const float* x, const float* w, const float* b, void* y, int rows, int d, float eps,
                           int out_format, wenc_stream_t stream) {
  g_last_error.clear();
  if (!x || !w || !b || !y) return fail(WENC_ERR_INVALID_ARG, "x/w/b/y is NULL");
  if (rows < 1) return fail(WENC_ERR_INVALID_ARG, "rows must be >= 1");
  if (!wenc_host::layernorm_supported(d)) return fail(WENC_ERR_UNSUPPORTED, "d %d: a multiple of 128 up to 2048", d);
  if (!(eps >= 0.0f)) return fail(WENC_ERR_INVALID_ARG, "eps must be >= 0");
  if (!aligned16(x) || !aligned16(w) || !aligned16(b) || !aligned16(y))
    return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (out_format < 0 || out_format > 2) return fail(WENC_ERR_INVALID_ARG, "out_format %d unknown", out_format);
  cudaError_t e = wenc_host::launch_layernorm(x, w, b, y, rows, d, eps, out_format, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "layernorm launch");
  return WENC_OK;
}

wenc_status wenc_linear(const uint16_t* A, const uint16_t* W, const float* bias, const float* resid, void* out, int M,
                        int N, int K, int epilogue, wenc_stream_t stream) {
  g_last_error.clear();
  if (!A || !W || !bias || !out) return fail(WENC_ERR_INVALID_ARG, "A/W/bias/out is NULL");
  if (epilogue < 0 || epilogue > 2) return fail(WENC_ERR_INVALID_ARG, "epilogue %d unknown", epilogue);
  if (epilogue == WENC_EPI_BIAS_RESID_F32 && !resid) return fail(WENC_ERR_INVALID_ARG, "resid is NULL");
  if (M < 1) return fail(WENC_ERR_INVALID_ARG, "M must be >= 1");
  const int bn = wenc_host::gemm_pick_bn(N);
  if (bn == 0) return fail(WENC_ERR_UNSUPPORTED, "N %d: must be a multiple of 128", N);
  if (K < 64 || K % 64 != 0) return fail(WENC_ERR_UNSUPPORTED, "K %d: must be a positive multiple of 64", K);
  if (!aligned16(A) || !aligned16(W) || !aligned16(bias) || !aligned16(out) || (resid && !aligned16(resid)))
    return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  std::string why;
  if (!device_is_sm103(&why)) return fail(WENC_ERR_UNSUPPORTED, "%s", why.c_str());
  uint32_t* err = global_error_word(&why);
  if (!err) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  CUtensorMap ta, tw, tw_h;
  bool ok = wenc_host::make_tmap_2d_bf16(&ta, A, K, M, size_t(K) * 2, 64, wenc_host::kGemmBM, &why) &&
            wenc_host::make_tmap_2d_bf16(&tw, W, K, N, size_t(K) * 2, 64, bn, &why) &&
            wenc_host::make_tmap_2d_bf16(&tw_h, W, K, N, size_t(K) * 2, 64, bn / 2, &why);
  if (!ok) return fail(WENC_ERR_INVALID_ARG, "%s", why.c_str());
  cudaError_t e = wenc_host::launch_gemm(ta, tw, M, N, K, bn, epilogue, bias, resid, out, err, sm_count(),
                                         reinterpret_cast<cudaStream_t>(stream), false, 0, wenc_host::GemmExtra(),
                                         &tw_h);
  if (e != cudaSuccess) return cuda_fail(e, "linear launch");
  return WENC_OK;
}

wenc_status wenc_linear_tf32(const float* A, const float* W, const float* bias, const float* resid, float* out, int M,
                             int N, int K, int epilogue, wenc_stream_t stream) {
  g_last_error.clear();
  if (!A || !W || !bias || !out) return fail(WENC_ERR_INVALID_ARG, "A/W/bias/out is NULL");
  if (epilogue < 0 || epilogue > 2) return fail(WENC_ERR_INVALID_ARG, "epilogue %d unknown", epilogue);
  if (epilogue == WENC_EPI_BIAS_RESID_F32 && !resid) return fail(WENC_ERR_INVALID_ARG, "resid is NULL");
  if (M < 1) return fail(WENC_ERR_INVALID_ARG, "M must be >= 1");
  const int bn = wenc_host::gemm_pick_bn(N);
  if (bn == 0) return fail(WENC_ERR_UNSUPPORTED, "N %d: must be a multiple of 128", N);
  if (K < 32 || K % 32 != 0) return fail(WENC_ERR_UNSUPPORTED, "K %d: must be a positive multiple of 32", K);
  if (!aligned16(A) || !aligned16(W) || !aligned16(bias) || !aligned16(out) || (resid && !aligned16(resid)))
    return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  std::string why;
  if (!device_is_sm103(&why)) return fail(WENC_ERR_UNSUPPORTED, "%s", why.c_str());
  uint32_t* err = global_error_word(&why);
  if (!err) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  CUtensorMap ta, tw;
  bool ok = wenc_host::make_tmap_2d_f32(&ta, A, K, M, size_t(K) * 4, 32, wenc_host::kGemmBM, &why) &&
            wenc_host::make_tmap_2d_f32(&tw, W, K, N, size_t(K) * 4, 32, bn, &why);
  if (!ok) return fail(WENC_ERR_INVALID_ARG, "%s", why.c_str());
  cudaError_t e = wenc_host::launch_gemm(ta, tw, M, N, K, bn, epilogue, bias, resid, out, err, sm_count(),
                                         reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "linear launch");
  return WENC_OK;
}

wenc_status wenc_attention_tf32(const float* q, const float* k, const float* v, float* out, int B, int T, int H, int hd,
                                wenc_stream_t stream) {
  g_last_error.clear();
  if (!q || !k || !v || !out) return fail(WENC_ERR_INVALID_ARG, "q/k/v/out is NULL");
  if (B < 1 || T < 1 || H < 1) return fail(WENC_ERR_INVALID_ARG, "B, T, H must be >= 1");
  if (hd != 64) return fail(WENC_ERR_UNSUPPORTED, "head_dim %d: only 64 is implemented", hd);
  if (T > (1 << 20)) return fail(WENC_ERR_UNSUPPORTED, "T %d too large", T);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  std::string why;
  if (!device_is_sm103(&why)) return fail(WENC_ERR_UNSUPPORTED, "%s", why.c_str());
  uint32_t* err = global_error_word(&why);
  if (!err) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  const uint64_t row = uint64_t(H) * 64;
  CUtensorMap tq, tk, tv;
  bool ok = wenc_host::make_tmap_3d_f32(&tq, q, row, T, B, row * 4, row * 4 * T, 32, wenc_host::kAttnTf32BQ, &why) &&
            wenc_host::make_tmap_3d_f32(&tk, k, row, T, B, row * 4, row * 4 * T, 32, wenc_host::kAttnTf32BKV, &why) &&
            wenc_host::make_tmap_3d_f32(&tv, v, row, T, B, row * 4, row * 4 * T, 32, wenc_host::kAttnTf32BKV, &why);
  if (!ok) return fail(WENC_ERR_INVALID_ARG, "%s", why.c_str());
  cudaError_t e = wenc_host::launch_attention_tf32(tq, tk, tv, 0, 0, 0, out, static_cast<int>(row), B, T, H, err,
                                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return WENC_OK;
}

wenc_status wenc_selftest_wait_timeout(wenc_stream_t stream) {
  g_last_error.clear();
  std::string why;
  uint32_t* err = global_error_word(&why);
  if (!err) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  stall_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return WENC_OK;
}

wenc_status wenc_selftest_gemm_pair_abort(const uint16_t* A, const uint16_t* W, const float* bias, uint16_t* out, int M,
                                          int N, int K, int stop_after, wenc_stream_t stream) {
  g_last_error.clear();
  if (!A || !W || !bias || !out) return fail(WENC_ERR_INVALID_ARG, "A/W/bias/out is NULL");
  if (M < 1 || stop_after < 0) return fail(WENC_ERR_INVALID_ARG, "M must be >= 1 and stop_after >= 0");
  if (N < 256 || N % 256 != 0) return fail(WENC_ERR_UNSUPPORTED, "N %d: the CTA-pair form needs a multiple of 256", N);
  if (K < 64 || K % 64 != 0) return fail(WENC_ERR_UNSUPPORTED, "K %d: must be a positive multiple of 64", K);
  if (!aligned16(A) || !aligned16(W) || !aligned16(bias) || !aligned16(out))
    return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  std::string why;
  if (!device_is_sm103(&why)) return fail(WENC_ERR_UNSUPPORTED, "%s", why.c_str());
  if (!wenc_host::gemm_pair_enabled()) return fail(WENC_ERR_UNSUPPORTED, "CTA-pair GEMMs are off (WENC_GEMM_PAIR=0)");
  uint32_t* err = global_error_word(&why);
  if (!err) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  CUtensorMap ta, tw, tw_h;
  bool ok = wenc_host::make_tmap_2d_bf16(&ta, A, K, M, size_t(K) * 2, 64, wenc_host::kGemmBM, &why) &&
            wenc_host::make_tmap_2d_bf16(&tw, W, K, N, size_t(K) * 2, 64, 256, &why) &&
            wenc_host::make_tmap_2d_bf16(&tw_h, W, K, N, size_t(K) * 2, 64, 128, &why);
  if (!ok) return fail(WENC_ERR_INVALID_ARG, "%s", why.c_str());
  wenc_host::GemmExtra ex;
  ex.stop_odd_after = stop_after;
  cudaError_t e = wenc_host::launch_gemm(ta, tw, M, N, K, 256, WENC_EPI_BIAS_BF16, bias, nullptr, out, err, sm_count(),
                                         reinterpret_cast<cudaStream_t>(stream), false, 0, ex, &tw_h);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return WENC_OK;
}

wenc_status wenc_selftest_attention_abort(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* out, int B,
                                          int T, int H, int stop_after, wenc_stream_t stream) {
  g_last_error.clear();
  if (!q || !k || !v || !out) return fail(WENC_ERR_INVALID_ARG, "q/k/v/out is NULL");
  if (B < 1 || T < 1 || H < 1 || stop_after < 0) return fail(WENC_ERR_INVALID_ARG, "B, T, H >= 1 and stop_after >= 0");
  if (T > (1 << 20)) return fail(WENC_ERR_UNSUPPORTED, "T %d too large", T);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  std::string why;
  if (!device_is_sm103(&why)) return fail(WENC_ERR_UNSUPPORTED, "%s", why.c_str());
  uint32_t* err = global_error_word(&why);
  if (!err) return fail(WENC_ERR_CUDA, "%s", why.c_str());
  const uint64_t row = uint64_t(H) * 64;
  CUtensorMap tq, tk, tv;
  bool ok = wenc_host::make_tmap_3d_bf16(&tq, q, row, T, B, row * 2, row * 2 * T, 64, wenc_host::kAttnBQ, &why) &&
            wenc_host::make_tmap_3d_bf16(&tk, k, row, T, B, row * 2, row * 2 * T, 64, wenc_host::kAttnBKV, &why) &&
            wenc_host::make_tmap_3d_bf16(&tv, v, row, T, B, row * 2, row * 2 * T, 64, wenc_host::kAttnBKV, &why);
  if (!ok) return fail(WENC_ERR_INVALID_ARG, "%s", why.c_str());
  cudaError_t e = wenc_host::launch_attention_main(tq, tk, tv, 0, 0, 0, out, static_cast<int>(row), B, T, H, err,
                                                   reinterpret_cast<cudaStream_t>(stream), 1, nullptr, nullptr,
                                                   stop_after);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return WENC_OK;
}

wenc_status wenc_selftest_gemm_schedule(int M, int N, int pair, int max_units, int* cover, int cover_len,
                                        int* unit_halves, int* units, int* halves) {
  g_last_error.clear();
  if (!cover || !units || !halves) return fail(WENC_ERR_INVALID_ARG, "cover/units/halves is NULL");
  const int r = wenc_host::gemm_schedule_cover(M, N, pair != 0, max_units, cover, cover_len, unit_halves, units,
                                               halves);
  if (r == -1) return fail(WENC_ERR_INVALID_ARG, "shape %d x %d (pair %d, %d units) unsupported or cover too short", M,
                           N, pair, max_units);
  if (r != 0) return fail(WENC_ERR_INVALID_ARG, "schedule produced a tile outside the launch");
  return WENC_OK;
}

wenc_status wenc_sync_status(wenc* h) {
  g_last_error.clear();
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  uint32_t word = 0;
  if (h) {
    word = *reinterpret_cast<volatile uint32_t*>(h->err_host);
    *reinterpret_cast<volatile uint32_t*>(h->err_host) = 0;
  } else {
    std::string why;
    if (!global_error_word(&why)) return fail(WENC_ERR_CUDA, "%s", why.c_str());
    e = cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word));
    if (e == cudaSuccess && word != 0) {
      const uint32_t zero = 0;
      e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
    }
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  }
  if (word != 0 && (word & 0xffu) == WENC_ERR_CUDA)
    return fail(WENC_ERR_CUDA, "an index check of the bounds-checked build failed (site %u)", (word >> 8) & 0xffu);
  if (word != 0)
    return fail(WENC_ERR_DEVICE_TIMEOUT, "device wait ran out (code %u, site %u)", word & 0xffu, (word >> 8) & 0xffu);
  return WENC_OK;
}

void wenc_destroy(wenc* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_handle(h);
}

}  // extern "C"
