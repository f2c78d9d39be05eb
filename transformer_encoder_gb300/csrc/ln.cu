// ln.cu -- LayerNorm over rows of the fp32 residual stream, and the weight-packing cast.
//
// y = (x - mean) / sqrt(var + eps) * w + b with the biased variance (inferencelayer 0.2.4
// src/whisper_gpu.rs, LN_SRC; turbospark-runtime 0.3.0 src/whisper/metal.rs, the
// encode_whisper_layer_norm calls of encode_layer and encode_partial; oxinfer 0.0.5
// src/whisper/model.rs, LayerNorm::apply_rows with LN_EPS).
//
// One warp per row: the row is read once from HBM with coalesced 16-byte loads and kept in
// registers, the mean and then the sum of squared deviations are reduced with shuffles (two
// passes over registers, one pass over memory), and the output is written as bf16 (feeding
// the next GEMM's TMA loads: LayerNorm and the operand cast fused), as fp32 rounded to TF32
// (the same for a TF32 GEMM) or as plain fp32 (the final LN).
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace {

constexpr int kRowsPerBlock = 8;  // 8 warps, one row each

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// NV = d / 128: float4 loads per lane. OUT: 0 = fp32, 1 = bf16, 2 = fp32 rounded to TF32.
template <int NV, int OUT>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    layernorm_kernel(const float* __restrict__ x, const float* __restrict__ w, const float* __restrict__ b,
                     void* __restrict__ y, int rows, float eps) {
  constexpr int D = NV * 128;
  wenc_dev::pdl_trigger();
  wenc_dev::pdl_wait();  // x from the previous kernel is complete from here on
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(row) * D);
  float4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = xr[lane + 32 * i];
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  const float mean = warp_sum(s) * (1.0f / D);
  float q = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const float a = v[i].x - mean, bb = v[i].y - mean, c = v[i].z - mean, d = v[i].w - mean;
    q += (a * a + bb * bb) + (c * c + d * d);
  }
  const float var = warp_sum(q) * (1.0f / D);
  const float rstd = 1.0f / sqrtf(var + eps);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  const float4* b4 = reinterpret_cast<const float4*>(b);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c4 = lane + 32 * i;
    const float4 ww = __ldg(w4 + c4), bb = __ldg(b4 + c4);
    float4 o;
    o.x = (v[i].x - mean) * rstd * ww.x + bb.x;
    o.y = (v[i].y - mean) * rstd * ww.y + bb.y;
    o.z = (v[i].z - mean) * rstd * ww.z + bb.z;
    o.w = (v[i].w - mean) * rstd * ww.w + bb.w;
    if constexpr (OUT == 1) {
      uint2 pk = make_uint2(wenc_dev::pack_bf16x2(o.x, o.y), wenc_dev::pack_bf16x2(o.z, o.w));
      reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + static_cast<size_t>(row) * D)[c4] = pk;
    } else {
      if constexpr (OUT == 2) {
        o.x = wenc_dev::round_tf32(o.x); o.y = wenc_dev::round_tf32(o.y);
        o.z = wenc_dev::round_tf32(o.z); o.w = wenc_dev::round_tf32(o.w);
      }
      reinterpret_cast<float4*>(static_cast<float*>(y) + static_cast<size_t>(row) * D)[c4] = o;
    }
  }
}

template <int NV>
cudaError_t launch_nv(const float* x, const float* w, const float* b, void* y, int rows, float eps, int out_fmt,
                      cudaStream_t stream) {
  const int grid = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const dim3 block(32 * kRowsPerBlock);
  if (out_fmt == 1) return wenc_host::launch_pdl(layernorm_kernel<NV, 1>, dim3(grid), block, 0, stream, x, w, b, y, rows, eps);
  if (out_fmt == 2) return wenc_host::launch_pdl(layernorm_kernel<NV, 2>, dim3(grid), block, 0, stream, x, w, b, y, rows, eps);
  return wenc_host::launch_pdl(layernorm_kernel<NV, 0>, dim3(grid), block, 0, stream, x, w, b, y, rows, eps);
}

// fp32 -> bf16, round to nearest with ties to even. Eight elements per thread and iteration
// (two 16-byte loads, one 16-byte store) when n and both pointers allow it, else one.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  const __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&a)) |
         (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&b)) << 16);
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst, size_t n, int vec8) {
  const size_t tid = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  if (vec8) {
    for (size_t i = tid; i < n / 8; i += stride) {
      const float4 a = reinterpret_cast<const float4*>(src)[2 * i];
      const float4 b = reinterpret_cast<const float4*>(src)[2 * i + 1];
      reinterpret_cast<uint4*>(dst)[i] =
          make_uint4(bf16x2_rn(a.x, a.y), bf16x2_rn(a.z, a.w), bf16x2_rn(b.x, b.y), bf16x2_rn(b.z, b.w));
    }
    return;
  }
  for (size_t i = tid; i < n; i += stride) {
    __nv_bfloat16 v = __float2bfloat16_rn(src[i]);
    dst[i] = *reinterpret_cast<uint16_t*>(&v);
  }
}

// Weight packing for the TF32 path: fp32 matrices are rounded to TF32 (nearest, ties away
// from zero); bf16 matrices are widened, which is exact (bf16 has fewer mantissa bits).
__global__ void to_tf32_kernel(const void* __restrict__ src, int src_bf16, float* __restrict__ dst, size_t n,
                               int vec4) {
  const size_t tid = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  if (vec4 && !src_bf16) {  // four fp32 elements per thread and iteration
    for (size_t i = tid; i < n / 4; i += stride) {
      const float4 a = reinterpret_cast<const float4*>(src)[i];
      reinterpret_cast<float4*>(dst)[i] = make_float4(wenc_dev::round_tf32(a.x), wenc_dev::round_tf32(a.y),
                                                      wenc_dev::round_tf32(a.z), wenc_dev::round_tf32(a.w));
    }
    return;
  }
  for (size_t i = tid; i < n; i += stride) {
    if (src_bf16)
      dst[i] = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(src)[i]) << 16);
    else
      dst[i] = wenc_dev::round_tf32(static_cast<const float*>(src)[i]);
  }
}

// The statistics a LayerNorm-folded GEMM needs, for a block's input rows (the BF16 forward's
// first block; later blocks get them from the residual epilogue of the GEMM before): one warp
// per row writes the row as bf16 (the GEMM operand) and the (mean, M2) of each SEG-column
// segment, computed exactly as that epilogue does (statistics of 32-column chunks, merged in
// column order), so the two give the same bits.
template <int NV, int SEG>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    row_stats_kernel(const float* __restrict__ x, uint16_t* __restrict__ xb, float2* __restrict__ stats, int rows) {
  constexpr int D = NV * 128;
  constexpr int CPS = SEG / 32;  // 32-column chunks per segment
  wenc_dev::pdl_trigger();
  wenc_dev::pdl_wait();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(row) * D);
  float4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = xr[lane + 32 * i];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    reinterpret_cast<uint2*>(xb + static_cast<size_t>(row) * D)[lane + 32 * i] =
        make_uint2(wenc_dev::pack_bf16x2(v[i].x, v[i].y), wenc_dev::pack_bf16x2(v[i].z, v[i].w));
    // columns 128 i + 32 m .. +31 are chunk m, held by lanes 8 m .. 8 m + 7
    float cm, cq;
    wenc_dev::chunk_stats32(v[i], cm, cq);
#pragma unroll
    for (int sg = 0; sg < 128 / SEG; ++sg) {
      float mean = 0.0f, m2 = 0.0f;
#pragma unroll
      for (int c = 0; c < CPS; ++c) {
        const int src = 8 * (sg * CPS + c);
        wenc_dev::chunk_merge32(mean, m2, __shfl_sync(0xffffffffu, cm, src), __shfl_sync(0xffffffffu, cq, src), c);
      }
      if (lane == 0) stats[static_cast<size_t>(row) * (D / SEG) + i * (128 / SEG) + sg] = make_float2(mean, m2);
    }
  }
}

template <int NV>
cudaError_t launch_row_stats_nv(const float* x, uint16_t* xb, float2* stats, int rows, int seg, cudaStream_t stream) {
  const int grid = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const dim3 block(32 * kRowsPerBlock);
  if (seg == 128) return wenc_host::launch_pdl(row_stats_kernel<NV, 128>, dim3(grid), block, 0, stream, x, xb, stats, rows);
  if (seg == 64) return wenc_host::launch_pdl(row_stats_kernel<NV, 64>, dim3(grid), block, 0, stream, x, xb, stats, rows);
  return cudaErrorInvalidValue;
}

// LayerNorm folded into the GEMM that follows it, at set-up: one block per output row n of
// W [n_out, k] (fp32 or bf16), with the LayerNorm's weight ln_w and shift ln_b [k]:
//   wp[n, j] = bf16(W[n, j] ln_w[j])           the GEMM's operand
//   colsum[n] = sum_j wp[n, j]                  (of the rounded values the GEMM multiplies)
//   bias_out[n] = sum_j W[n, j] ln_b[j] + bias[n]   (bias may be NULL: zero)
// so that LN(x) W^T + bias = rstd (x wp^T - mean colsum) + bias_out.
__global__ void __launch_bounds__(256) fold_ln_kernel(const void* __restrict__ w, int w_bf16, const float* __restrict__ ln_w,
                                                      const float* __restrict__ ln_b, const float* __restrict__ bias,
                                                      uint16_t* __restrict__ wp, float* __restrict__ colsum,
                                                      float* __restrict__ bias_out, int k) {
  const size_t n = blockIdx.x;
  float s = 0.0f, c = 0.0f;
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const size_t idx = n * k + j;
    const float wv = w_bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(w)[idx]) << 16)
                            : static_cast<const float*>(w)[idx];
    const __nv_bfloat16 hv = __float2bfloat16_rn(wv * ln_w[j]);  // nearest, ties to even
    wp[idx] = *reinterpret_cast<const uint16_t*>(&hv);
    s += __bfloat162float(hv);
    c = fmaf(wv, ln_b[j], c);
  }
  __shared__ float red[2][8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    c += __shfl_xor_sync(0xffffffffu, c, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = s;
    red[1][threadIdx.x >> 5] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float ts = 0.0f, tc = 0.0f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) {
      ts += red[0][i];
      tc += red[1][i];
    }
    colsum[n] = ts;
    bias_out[n] = tc + (bias ? bias[n] : 0.0f);
  }
}

}  // namespace

namespace wenc_host {

bool layernorm_supported(int d) { return d > 0 && d % 128 == 0 && d / 128 <= 16; }

cudaError_t launch_layernorm(const float* x, const float* w, const float* b, void* y, int rows, int d, float eps,
                             int out_fmt, cudaStream_t stream) {
  if (out_fmt < 0 || out_fmt > 2) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  switch (d / 128) {
#define WENC_LN_CASE(N) \
  case N: return launch_nv<N>(x, w, b, y, rows, eps, out_fmt, stream);
    WENC_LN_CASE(1) WENC_LN_CASE(2) WENC_LN_CASE(3) WENC_LN_CASE(4) WENC_LN_CASE(5) WENC_LN_CASE(6)
    WENC_LN_CASE(7) WENC_LN_CASE(8) WENC_LN_CASE(9) WENC_LN_CASE(10) WENC_LN_CASE(11) WENC_LN_CASE(12)
    WENC_LN_CASE(13) WENC_LN_CASE(14) WENC_LN_CASE(15) WENC_LN_CASE(16)
#undef WENC_LN_CASE
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_row_stats(const float* x, uint16_t* xb, float2* stats, int rows, int d, int seg, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  switch (d / 128) {
#define WENC_RS_CASE(N) \
  case N: return launch_row_stats_nv<N>(x, xb, stats, rows, seg, stream);
    WENC_RS_CASE(1) WENC_RS_CASE(2) WENC_RS_CASE(3) WENC_RS_CASE(4) WENC_RS_CASE(5) WENC_RS_CASE(6)
    WENC_RS_CASE(7) WENC_RS_CASE(8) WENC_RS_CASE(9) WENC_RS_CASE(10) WENC_RS_CASE(11) WENC_RS_CASE(12)
    WENC_RS_CASE(13) WENC_RS_CASE(14) WENC_RS_CASE(15) WENC_RS_CASE(16)
#undef WENC_RS_CASE
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fold_ln(const void* w, bool w_bf16, const float* ln_w, const float* ln_b, const float* bias,
                           uint16_t* wp, float* colsum, float* bias_out, int n_out, int k, cudaStream_t stream) {
  if (n_out <= 0) return cudaSuccess;
  fold_ln_kernel<<<n_out, 256, 0, stream>>>(w, w_bf16 ? 1 : 0, ln_w, ln_b, bias, wp, colsum, bias_out, k);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const bool vec8 = n % 8 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const size_t blocks = ((vec8 ? n / 8 : n) + 255) / 256;
  f32_to_bf16_kernel<<<static_cast<unsigned>(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, stream>>>(src, dst, n,
                                                                                                   vec8 ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_to_tf32(const void* src, bool src_bf16, float* dst, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const bool vec4 = !src_bf16 && n % 4 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const size_t blocks = ((vec4 ? n / 4 : n) + 255) / 256;
  to_tf32_kernel<<<static_cast<unsigned>(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, stream>>>(
      src, src_bf16 ? 1 : 0, dst, n, vec4 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace wenc_host
