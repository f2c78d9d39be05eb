// gemm.cu -- the block's four contractions on the 5th-generation tensor cores.
//
// C[M, N] = A[M, K] . W[N, K]^T with the epilogue fused (the matmul_bias step of
// turbospark-runtime src/whisper/metal.rs encode_layer, with its separate add and
// gelu_erf passes folded in; inferencelayer src/whisper_gpu.rs WhisperEncoderGpu::forward
// fuses bias + GELU into its fc1 GEMM the same way):
//   QKV:      bf16 out = A W^T + b             (b's K slot is zero)
//   fc1:      bf16 out = GELU_erf(A W^T + b)
//   out, fc2: f32  out = resid + (A W^T + b)   (the residual add, in place on x)
//
// Design (sm_103a): persistent CTAs, one per SM, walk 128 x BN output tiles. Warp 0 is the
// TMA producer (A and W tiles, 128-byte swizzle, a STAGES-deep mbarrier ring); warp 1
// allocates TMEM and one of its threads issues tcgen05.mma (128 x BN x 16, bf16 in, fp32
// accumulate) into one of two TMEM accumulators; warps 2-5 drain the other accumulator
// (tcgen05.ld -> bias / GELU / residual -> global) while the next tile is being computed.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace {

using namespace wenc_dev;

constexpr int BM = wenc_host::kGemmBM;
constexpr int BK = wenc_host::kGemmBK;
constexpr int kEpiWarps = 8;                // two warps per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer warp, MMA warp, epilogue warps

template <int BN>
struct GemmCfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two fp32 accumulators of BN columns
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 5;
  static constexpr size_t SMEM = 1024 /*align slack*/ + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
};

__device__ __forceinline__ float gelu_erf(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }

template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const uint32_t (&acc)[32], const float4 (&rr)[8],
                                               const float* __restrict__ bias, void* out, size_t row_off, int col0) {
  const float4* b4 = reinterpret_cast<const float4*>(bias + col0);
  if constexpr (EPI == 2) {
    float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(out) + row_off + col0);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 bb = __ldg(b4 + j);
      float4 v;
      v.x = rr[j].x + (__uint_as_float(acc[4 * j + 0]) + bb.x);
      v.y = rr[j].y + (__uint_as_float(acc[4 * j + 1]) + bb.y);
      v.z = rr[j].z + (__uint_as_float(acc[4 * j + 2]) + bb.z);
      v.w = rr[j].w + (__uint_as_float(acc[4 * j + 3]) + bb.w);
      o4[j] = v;
    }
  } else {
    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 bb = __ldg(b4 + j);
      float v0 = __uint_as_float(acc[4 * j + 0]) + bb.x;
      float v1 = __uint_as_float(acc[4 * j + 1]) + bb.y;
      float v2 = __uint_as_float(acc[4 * j + 2]) + bb.z;
      float v3 = __uint_as_float(acc[4 * j + 3]) + bb.w;
      if constexpr (EPI == 1) {
        v0 = gelu_erf(v0); v1 = gelu_erf(v1); v2 = gelu_erf(v2); v3 = gelu_erf(v3);
      }
      packed[2 * j] = pack_bf16x2(v0, v1);
      packed[2 * j + 1] = pack_bf16x2(v2, v3);
    }
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + row_off + col0);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
  }
}

// Residual row segment of 32 fp32 values (128 bytes) into registers.
__device__ __forceinline__ void load_resid(float4 (&rr)[8], const float* resid, size_t off) {
  const float4* r4 = reinterpret_cast<const float4*>(resid + off);
#pragma unroll
  for (int j = 0; j < 8; ++j) rr[j] = r4[j];
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, int M, int N,
                   int K, const float* __restrict__ bias, const float* resid, void* out, uint32_t* err) {
  using C = GemmCfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * C::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, err};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = (M + BM - 1) / BM;
  const int n_tiles = N / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int k_blocks = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const int m0 = (tile / n_tiles) * BM;
      const int n0 = (tile % n_tiles) * BN;
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc, 1)) { ok = false; break; }
        mbar_arrive_expect_tx(full_bar(stage), C::STAGE_BYTES);
        tma_load_2d(sA + stage * C::A_BYTES, &tmA, full_bar(stage), kb * BK, m0);
        tma_load_2d(sB + stage * C::B_BYTES, &tmW, full_bar(stage), kb * BK, n0);
        issued_mask |= 1u << stage;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      // Error path: let the copies already issued land before the CTA exits.
      for (int s = 0; s < STAGES; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        mbar_wait_drain(full_bar(s), par);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- UMMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, wc, 2)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, wc, 3)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_base = sA + stage * C::A_BYTES;
        const uint32_t b_base = sB + stage * C::B_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t ad = sdesc_sw128(a_base + k * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(b_base + k * 32, 16, 1024);
          umma_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
        }
        umma_commit(empty_bar(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      umma_commit(tfull_bar(acc));
    }
    // Every UMMA issued by this thread completes before TMEM is released.
    umma_commit(drain_bar);
    mbar_wait_drain(drain_bar, 0);
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> registers -> global
    // Eight warps: warp w reads TMEM lane quadrant w % 4 (rows 32q..32q+31 of the tile) and
    // one half of the tile's columns. Each thread owns one output row. For the residual
    // epilogue the row's fp32 residual is loaded two 32-column chunks ahead, starting
    // before the accumulator is ready, so that enough bytes are in flight to cover HBM
    // latency; the TMEM buffer is released as soon as its last chunk has been read.
    constexpr int CH = BN / 64;  // 32-column chunks per warp
    const int quad = warp & 3;
    const int col_half = (warp - 2) >> 2;
    const int row_in_tile = quad * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int m0 = (tile / n_tiles) * BM;
      const int n0 = (tile % n_tiles) * BN;
      const int row = m0 + row_in_tile;
      const bool live = row < M;
      const int c0 = n0 + col_half * (BN / 2);
      const size_t row_off = static_cast<size_t>(row) * N;
      float4 rb[2][8];
      if constexpr (EPI == 2) {
        if (live) {
          load_resid(rb[0], resid, row_off + c0);
          if (CH > 1) load_resid(rb[1], resid, row_off + c0 + 32);
        }
      }
      if (!mbar_wait_warp(tfull_bar(acc), acc_phase, wc, 4)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN + col_half * (BN / 2);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
        if (c == CH - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
        if (live) epilogue_chunk<EPI>(r, rb[c & 1], bias, out, row_off, c0 + c * 32);
        if constexpr (EPI == 2) {
          if (live && c + 2 < CH) load_resid(rb[c & 1], resid, row_off + c0 + (c + 2) * 32);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int EPI>
cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmW, int M, int N, int K, const float* bias,
                       const float* resid, void* out, uint32_t* err, int num_sms, cudaStream_t stream) {
  using C = GemmCfg<BN>;
  auto kern = gemm_tc_kernel<BN, EPI>;
  static int configured_device = -1;  // attribute is per device; cheap to repeat
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int tiles = ((M + BM - 1) / BM) * (N / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  kern<<<grid, kThreads, C::SMEM, stream>>>(tmA, tmW, M, N, K, bias, resid, out, err);
  return cudaGetLastError();
}

}  // namespace

namespace wenc_host {

int gemm_pick_bn(int N) {
  if (N % 256 == 0) return 256;
  if (N % 128 == 0) return 128;
  return 0;
}

cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmW, int M, int N, int K, int bn, int epilogue,
                        const float* bias, const float* resid, void* out, uint32_t* err, int num_sms,
                        cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
#define WENC_GEMM_CASE(BNV, EPIV) \
  if (bn == BNV && epilogue == EPIV) return launch_one<BNV, EPIV>(tmA, tmW, M, N, K, bias, resid, out, err, num_sms, stream);
  WENC_GEMM_CASE(256, 0)
  WENC_GEMM_CASE(256, 1)
  WENC_GEMM_CASE(256, 2)
  WENC_GEMM_CASE(128, 0)
  WENC_GEMM_CASE(128, 1)
  WENC_GEMM_CASE(128, 2)
#undef WENC_GEMM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace wenc_host
