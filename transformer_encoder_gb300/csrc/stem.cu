// stem.cu -- the convolutional stem's data movement: unfolding a signal for a kernel-3
// convolution, and the convolution weights in the matching order.
//
// The stem (turbospark-runtime 0.3.0 src/whisper/metal.rs, encode_partial: conv1 with stride 1
// and padding 1, conv2 with stride 2 and padding 1, exact-erf GELU, positional rows; oxinfer
// 0.0.5 src/whisper/model.rs, WhisperModel::encode) runs each convolution as one tcgen05 GEMM:
// y[t, o] = b[o] + sum_{j, i} w[o, i, j] x[stride*t + j - 1, i] is the product of the unfolded
// signal A[t, j*C + i] = x[stride*t + j - 1, i] with the weight reordered to Wp[o, j*C + i].
// These two kernels build A (per call) and Wp (once, at set-up); the GEMM's epilogue adds the
// bias, the GELU and, for conv2, the positional row. The unfolded signal is written once and read
// once by the GEMM: 3x the input bytes (the stem is under 1% of the encoder's work).
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace {

__device__ __forceinline__ void load8(const void* x, bool x_f32, size_t off, float (&v)[8], uint4& raw) {
  if (x_f32) {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + off + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    raw = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off);
  }
}

// One warp per unfolded row (window b, output position t): the row's source frames are found
// once, and the lanes walk its 8-element chunks (chunk c: tap c / (C/8), channels 8 (c % (C/8))).
template <bool X_F32, bool A_TF32>
__global__ void __launch_bounds__(256) unfold3_kernel(const void* __restrict__ x, void* __restrict__ a, int t_in,
                                                      int t_out, int C, int stride, int k_pad, int rows) {
  wenc_dev::pdl_trigger();
  wenc_dev::pdl_wait();  // x from the previous kernel is complete from here on
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int cpr = k_pad / 8;  // 8-element chunks per unfolded row
  const int cpt = C / 8;      // chunks per tap
  for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += warps) {
    const int b = row / t_out;
    const int t = row - b * t_out;
    const size_t row_off = static_cast<size_t>(row) * k_pad;
    for (int c = lane; c < cpr; c += 32) {
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);  // bf16 input passed through unchanged
      if (c < 3 * cpt) {
        const int j = c / cpt;
        const int i = (c - j * cpt) * 8;
        const int src = stride * t + j - 1;
        if (src >= 0 && src < t_in) load8(x, X_F32, (static_cast<size_t>(b) * t_in + src) * C + i, v, raw);
      }
      const size_t off = row_off + static_cast<size_t>(c) * 8;
      if constexpr (A_TF32) {
        float* dst = static_cast<float*>(a) + off;
        *reinterpret_cast<float4*>(dst) = make_float4(wenc_dev::round_tf32(v[0]), wenc_dev::round_tf32(v[1]),
                                                      wenc_dev::round_tf32(v[2]), wenc_dev::round_tf32(v[3]));
        *reinterpret_cast<float4*>(dst + 4) = make_float4(wenc_dev::round_tf32(v[4]), wenc_dev::round_tf32(v[5]),
                                                          wenc_dev::round_tf32(v[6]), wenc_dev::round_tf32(v[7]));
      } else if constexpr (X_F32) {
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a) + off) =
            make_uint4(wenc_dev::pack_bf16x2(v[0], v[1]), wenc_dev::pack_bf16x2(v[2], v[3]),
                       wenc_dev::pack_bf16x2(v[4], v[5]), wenc_dev::pack_bf16x2(v[6], v[7]));
      } else {
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a) + off) = raw;
      }
    }
  }
}

// wp[o, j*c_in + i] = w[o, i, j]; zeros beyond 3*c_in. Runs once per set-up.
__global__ void conv_weight_kernel(const void* __restrict__ w, int w_bf16, void* __restrict__ wp, int wp_tf32,
                                   int c_out, int c_in, int k_pad) {
  const long long total = static_cast<long long>(c_out) * k_pad;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long o = idx / k_pad;
    const int col = static_cast<int>(idx % k_pad);
    float v = 0.0f;
    if (col < 3 * c_in) {
      const int j = col / c_in, i = col % c_in;
      const size_t src = (static_cast<size_t>(o) * c_in + i) * 3 + j;
      v = w_bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(w)[src]) << 16)
                 : static_cast<const float*>(w)[src];
    }
    if (wp_tf32) {
      static_cast<float*>(wp)[idx] = wenc_dev::round_tf32(v);
    } else {
      const __nv_bfloat16 hv = __float2bfloat16_rn(v);  // nearest, ties to even
      static_cast<uint16_t*>(wp)[idx] = *reinterpret_cast<const uint16_t*>(&hv);
    }
  }
}

}  // namespace

namespace wenc_host {

cudaError_t launch_unfold3(const void* x, bool x_f32, void* a, bool a_tf32, int B, int t_in, int C, int stride,
                           int k_pad, cudaStream_t stream) {
  if (C % 8 != 0 || k_pad % 8 != 0 || k_pad < 3 * C || (stride != 1 && stride != 2)) return cudaErrorInvalidValue;
  if (!x_f32 && a_tf32) return cudaErrorInvalidValue;  // bf16 input only feeds a bf16 GEMM
  const int t_out = (t_in + 2 - 3) / stride + 1;
  const long long rows = static_cast<long long>(B) * t_out;
  if (rows <= 0) return cudaSuccess;
  if (rows > (1LL << 30)) return cudaErrorInvalidValue;
  const long long want = (rows + 7) / 8;  // 8 rows (warps) per block
  const dim3 grid(static_cast<unsigned>(want < 152 * 16 ? want : 152 * 16));
  const int r = static_cast<int>(rows);
  if (x_f32 && a_tf32)
    return launch_pdl(unfold3_kernel<true, true>, grid, dim3(256), 0, stream, x, a, t_in, t_out, C, stride, k_pad, r);
  if (x_f32)
    return launch_pdl(unfold3_kernel<true, false>, grid, dim3(256), 0, stream, x, a, t_in, t_out, C, stride, k_pad, r);
  return launch_pdl(unfold3_kernel<false, false>, grid, dim3(256), 0, stream, x, a, t_in, t_out, C, stride, k_pad, r);
}

cudaError_t launch_conv_weight(const void* w, bool w_bf16, void* wp, bool wp_tf32, int c_out, int c_in, int k_pad,
                               cudaStream_t stream) {
  if (k_pad < 3 * c_in) return cudaErrorInvalidValue;
  const long long total = static_cast<long long>(c_out) * k_pad;
  if (total <= 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  conv_weight_kernel<<<static_cast<unsigned>(want < 4096 ? want : 4096), 256, 0, stream>>>(
      w, w_bf16 ? 1 : 0, wp, wp_tf32 ? 1 : 0, c_out, c_in, k_pad);
  return cudaGetLastError();
}

}  // namespace wenc_host
