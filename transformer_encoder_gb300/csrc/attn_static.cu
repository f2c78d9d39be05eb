// attn_static.cu -- attention for callers that cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc at all: a host that hands out device
// memory only from its own fixed pool, a runtime that forbids allocation once it is serving,
// or code running where an allocation would synchronise the device or break a recorded work
// sequence. wenc_attention_static serves them: it computes the same attention as
// wenc_attention, with the keys split among several CTAs per query pair and the partial results
// merged by a second kernel, and keeps those partial results in a buffer that is part of the
// library's own device image instead of memory allocated per call.
//
// The buffer below is a file-scope device array of kStaticScratchBytes. Every GPU that loads
// the library holds it until the process exits. In host code its name stands for a host-side
// shadow, not a device address, so the kernels are never handed that name: on the first call
// on each device (with that device current) cudaGetSymbolAddress returns the device address,
// which is cached per device and passed to the kernels.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "launch.h"
#include "wenc.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB

// Partial numerators first, then the (max, sum) pairs; both regions start 256-byte aligned.
static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_attn_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

using namespace wenc_host;

// Defined in api.cu: status helpers and the handle-less device error word.
wenc_status wenc_internal_fail(wenc_status s, const char* msg);
void wenc_internal_clear_error();
uint32_t* wenc_internal_error_word(std::string* why);
bool wenc_internal_is_sm103(std::string* why);
int wenc_internal_sm_count();

extern "C" WENC_API size_t wenc_attention_static_capacity(void) { return kStaticScratchBytes; }

extern "C" WENC_API wenc_status wenc_attention_static(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                                      uint16_t* out, int B, int T, int H, int hd,
                                                      wenc_stream_t stream) {
  wenc_internal_clear_error();  // a successful call leaves no message from an earlier failure
  if (!q || !k || !v || !out) return wenc_internal_fail(WENC_ERR_INVALID_ARG, "q/k/v/out is NULL");
  if (B < 1 || T < 1 || H < 1) return wenc_internal_fail(WENC_ERR_INVALID_ARG, "B, T, H must be >= 1");
  if (hd != 64) return wenc_internal_fail(WENC_ERR_UNSUPPORTED, "head_dim must be 64");
  if (T > (1 << 20)) return wenc_internal_fail(WENC_ERR_UNSUPPORTED, "T too large");
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(out))
    return wenc_internal_fail(WENC_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  // Split the keys the way a handle would for this shape, and at least in two whenever there
  // are two key tiles, so that the partial results always go through the static buffer.
  const int n_kv = (T + kAttnBKV - 1) / kAttnBKV;
  int n_splits = attention_pick_splits(B, T, H, wenc_internal_sm_count());
  if (n_splits < 2 && n_kv >= 2) n_splits = 2;
  const size_t need = attention_partial_bytes(B, T, H, n_splits);
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "B*H*T = %lld needs %zu bytes of partial results, more than the %zu-byte static buffer; "
             "use wenc_attention (no scratch) or fewer windows/heads per call",
             static_cast<long long>(B) * H * T, need, kStaticScratchBytes);
    return wenc_internal_fail(WENC_ERR_INVALID_ARG, msg);
  }
  std::string why;
  if (!wenc_internal_is_sm103(&why)) return wenc_internal_fail(WENC_ERR_UNSUPPORTED, why.c_str());
  uint32_t* err = wenc_internal_error_word(&why);
  if (!err) return wenc_internal_fail(WENC_ERR_CUDA, why.c_str());
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return wenc_internal_fail(WENC_ERR_CUDA, cudaGetErrorString(e));
  }
  const size_t rows = static_cast<size_t>(n_splits) * B * H * T;
  float* part_o = static_cast<float*>(scratch);
  float2* part_ml = reinterpret_cast<float2*>(static_cast<unsigned char*>(scratch) +
                                              ((rows * kAttnHD * sizeof(float) + 255) & ~size_t(255)));
  const uint64_t row = uint64_t(H) * 64;
  CUtensorMap tq, tk, tv;
  const bool ok = make_tmap_3d_bf16(&tq, q, row, T, B, row * 2, row * 2 * T, 64, kAttnBQ, &why) &&
                  make_tmap_3d_bf16(&tk, k, row, T, B, row * 2, row * 2 * T, 64, kAttnBKV, &why) &&
                  make_tmap_3d_bf16(&tv, v, row, T, B, row * 2, row * 2 * T, 64, kAttnBKV, &why);
  if (!ok) return wenc_internal_fail(WENC_ERR_INVALID_ARG, why.c_str());
  e = launch_attention(tq, tk, tv, 0, 0, 0, out, static_cast<int>(row), B, T, H, err,
                       reinterpret_cast<cudaStream_t>(stream), n_splits, part_o, part_ml);
  if (e != cudaSuccess) return wenc_internal_fail(WENC_ERR_CUDA, cudaGetErrorString(e));
  return WENC_OK;
}
