// attn.cu -- non-causal scaled-dot attention of one encoder window, fused (flash style).
//
// What it computes (inferencelayer 0.2.4 src/whisper_gpu.rs, VANILLA_ATTN; turbospark-runtime
// 0.3.0 src/whisper/metal.rs, encode_layer): for every window b, head h and query row i,
//   s_j = (q_i . k_j) * hd^-0.5 over all T keys,  p = softmax(s),  o_i = sum_j p_j v_j.
// No mask beyond the window's own length, no positional term.
//
// How (sm_103a): one CTA per (128-query tile, head, window), two CTAs per SM. Warp 0 streams
// K/V tiles of 64 keys with TMA into a 3-deep ring; one thread of warp 1 issues
// S = Q K^T (128 x 64 x 64) into one of two TMEM score buffers and, once the softmax warps
// have written P, O += P V (128 x 64 x 64, V read MN-major) into a TMEM accumulator; S[j+2]
// is queued right behind PV[j]. Warps 2-5 own one query row per thread: they read S from
// TMEM, keep the running maximum and denominator in registers (the online-softmax recurrence
// of VANILLA_ATTN, in base 2 with hd^-0.5*log2(e) folded in), write P as bf16 into one of two
// 128-byte-swizzled shared-memory buffers and, only when the running maximum grows by more
// than 2^8, wait for the previous PV and rescale O in TMEM. No T x T score buffer exists.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"

namespace {

using namespace wenc_dev;

constexpr int BQ = wenc_host::kAttnBQ;    // query rows per CTA
constexpr int BKV = wenc_host::kAttnBKV;  // keys per tile
constexpr int HD = 64;
constexpr int NST = 3;  // K/V ring depth
constexpr int kThreads = 192;

constexpr uint32_t Q_BYTES = BQ * HD * 2;    // 16 KB
constexpr uint32_t P_BYTES = BQ * BKV * 2;   // 16 KB
constexpr uint32_t KV_BYTES = BKV * HD * 2;  // 8 KB per K or V tile
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_P = OFF_Q + Q_BYTES;  // two P buffers
constexpr uint32_t OFF_K = OFF_P + 2 * P_BYTES;
constexpr uint32_t OFF_V = OFF_K + NST * KV_BYTES;
constexpr uint32_t OFF_BARS = OFF_V + NST * KV_BYTES;
// bars: q_full, kv_full[NST], kv_empty[NST], s_full[2], s_free[2], p_full[2], pv_done[2], drain
constexpr int NUM_BARS = 1 + 2 * NST + 9;
constexpr size_t SMEM = 1024 + OFF_BARS + NUM_BARS * 8 + 16;
constexpr uint32_t TMEM_COLS = 256;  // S buffers: columns 0..63 and 64..127; O: 128..191
// Grow the running maximum only when a tile's maximum exceeds it by more than this (log2
// units); otherwise keep it, so p <= 2^8 and O is rescaled rarely. The result is unchanged:
// numerator and denominator always use the same reference maximum.
constexpr float kRescaleThreshold = 8.0f;

__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, int q_col0, int k_col0, int v_col0,
                    uint16_t* __restrict__ out, int out_stride, int T, float scale_log2, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ = s0 + OFF_Q, sP = s0 + OFF_P, sK = s0 + OFF_K, sV = s0 + OFF_V;
  const uint32_t bar0 = s0 + OFF_BARS;
  const uint32_t q_full = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (1 + NST + s); };
  const uint32_t sb0 = bar0 + 8u * (1 + 2 * NST);
  auto s_full = [&](int b) { return sb0 + 8u * b; };
  auto s_free = [&](int b) { return sb0 + 16u + 8u * b; };
  auto p_full = [&](int b) { return sb0 + 32u + 8u * b; };
  auto pv_done = [&](int b) { return sb0 + 48u + 8u * b; };
  const uint32_t drain = sb0 + 64u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BARS + NUM_BARS * 8);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, err};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * BQ;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int n_kv = (T + BKV - 1) / BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_free(i), 4);  // one arrival per softmax warp
      mbar_init(p_full(i), 4);
      mbar_init(pv_done(i), 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto tS = [&](int b) { return tmem_base + 64u * b; };
  const uint32_t tO = tmem_base + 128;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    mbar_arrive_expect_tx(q_full, Q_BYTES);
    tma_load_3d(sQ, &tq, q_full, q_col0 + h * HD, q0, b);
    int issued = 0;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j % NST;
      const uint32_t ph = (j / NST) & 1;
      if (!mbar_wait(kv_empty(st), ph ^ 1u, wc, 11)) break;
      mbar_arrive_expect_tx(kv_full(st), 2 * KV_BYTES);
      tma_load_3d(sK + st * KV_BYTES, &tk, kv_full(st), k_col0 + h * HD, j * BKV, b);
      tma_load_3d(sV + st * KV_BYTES, &tv, kv_full(st), v_col0 + h * HD, j * BKV, b);
      issued = j + 1;
    }
    if (*abort_flag) {
      // Error path: let the copies already issued land before the CTA exits.
      mbar_wait_drain(q_full, 0);
      for (int j = (issued > NST ? issued - NST : 0); j < issued; ++j) mbar_wait_drain(kv_full(j % NST), (j / NST) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- UMMA issuer
    // Order on the tensor pipe: S0, S1, PV0, S2, PV1, S3, ... S[j+2] is queued right behind
    // PV[j], so a score tile is always ready before the softmax warps ask for it.
    constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV, false);  // B = K tile, K-major
    constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, HD, true);    // B = V tile, MN-major
    auto issue_s = [&](int j) -> bool {
      const int st = j % NST;
      if (!mbar_wait(kv_full(st), (j / NST) & 1, wc, 13)) return false;
      if (j >= 2 && !mbar_wait(s_free(j & 1), ((j - 2) >> 1) & 1, wc, 14)) return false;
      tc_fence_after();
      const uint32_t kb = sK + st * KV_BYTES;
#pragma unroll
      for (int k = 0; k < HD / 16; ++k)
        umma_bf16_ss(tS(j & 1), sdesc_sw128(sQ + k * 32, 16, 1024), sdesc_sw128(kb + k * 32, 16, 1024), idesc_s,
                     k > 0);
      umma_commit(s_full(j & 1));
      return true;
    };
    bool ok = mbar_wait(q_full, 0, wc, 12) && issue_s(0) && (n_kv < 2 || issue_s(1));
    for (int j = 0; ok && j < n_kv; ++j) {
      const int st = j % NST;
      if (!mbar_wait(p_full(j & 1), (j >> 1) & 1, wc, 16)) break;
      tc_fence_after();
      const uint32_t pb = sP + (j & 1) * P_BYTES;
      const uint32_t vb = sV + st * KV_BYTES;
#pragma unroll
      for (int k = 0; k < BKV / 16; ++k)
        umma_bf16_ss(tO, sdesc_sw128(pb + k * 32, 16, 1024), sdesc_sw128(vb + k * 2048, 1024, 1024), idesc_o,
                     (j > 0 || k > 0) ? 1u : 0u);
      umma_commit(pv_done(j & 1));
      umma_commit(kv_empty(st));
      if (j + 2 < n_kv) ok = issue_s(j + 2);
    }
    umma_commit(drain);
    mbar_wait_drain(drain, 0);
  } else if (warp >= 2) {
    // ---------------- softmax / correction / output: one query row per thread
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float m = -CUDART_INF_F;  // running maximum, in units of scale_log2
    float l = 0.0f;           // running denominator
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int pb = j & 1;  // S buffer and P buffer of this tile
      if (!mbar_wait_warp(s_full(pb), (j >> 1) & 1, wc, 17)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld_32x32b_x32(tS(pb) + lane_off, sr[0]);
      tmem_ld_32x32b_x32(tS(pb) + lane_off + 32, sr[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(pb));

      float sv[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) sv[c] = __uint_as_float(sr[c >> 5][c & 31]);
      const int valid = T - j * BKV;  // keys of this tile inside the window
      if (valid < BKV) {              // only a window's last tile can be partial (warp-uniform)
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = (c < valid) ? sv[c] : -CUDART_INF_F;
      }
      // Row maximum: four independent chains of three-input max.
      float mc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a = fmax3(sv[16 * k], sv[16 * k + 1], sv[16 * k + 2]);
#pragma unroll
        for (int e = 3; e < 15; e += 2) a = fmax3(a, sv[16 * k + e], sv[16 * k + e + 1]);
        mc[k] = fmaxf(a, sv[16 * k + 15]);
      }
      const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), mc[3]);
      const float mx_s = mx * scale_log2;
      const float m_new = (mx_s > m + kRescaleThreshold) ? mx_s : m;
      const float alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)

      // p = 2^(s * scale_log2 - m_new): packed fp32x2 FMA for the argument, packed adds for
      // the row sum; P is packed to bf16 pairs before waiting on the previous PV product.
      const uint64_t c2 = pack_f32x2(scale_log2, scale_log2);
      const uint64_t nm2 = pack_f32x2(-m_new, -m_new);
      uint64_t sum2a = pack_f32x2(0.0f, 0.0f), sum2b = sum2a;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a0, a1;
        unpack_f32x2(fma_f32x2(pack_f32x2(sv[2 * i], sv[2 * i + 1]), c2, nm2), a0, a1);
        const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
        if (i & 1) sum2b = add_f32x2(sum2b, pack_f32x2(p0, p1));
        else sum2a = add_f32x2(sum2a, pack_f32x2(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      float sa0, sa1, sb0, sb1;
      unpack_f32x2(sum2a, sa0, sa1);
      unpack_f32x2(sum2b, sb0, sb1);
      const float sum = (sa0 + sa1) + (sb0 + sb1);

      if (j > 0 && __any_sync(0xffffffffu, m_new != m)) {
        // The running maximum moved: O must hold every PV up to tile j-1 before it is rescaled.
        if (!mbar_wait_warp(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, wc, 18)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + lane_off + half * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x32(tO + lane_off + half * 32, o);
        }
        tmem_st_wait();
      } else if (j >= 2) {
        // P buffer pb was last read by PV[j-2].
        if (!mbar_wait_warp(pv_done(pb), ((j - 2) >> 1) & 1, wc, 20)) { ok = false; break; }
      }

      const uint32_t prow = sP + pb * P_BYTES + row * 128;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint32_t addr = prow + ((c8 ^ (row & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c8]), "r"(pk[4 * c8 + 1]),
                     "r"(pk[4 * c8 + 2]), "r"(pk[4 * c8 + 3])
                     : "memory");
      }
      l = l * alpha + sum;
      m = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(pb));
    }
    if (ok && mbar_wait_warp(pv_done((n_kv - 1) & 1), ((n_kv - 1) >> 1) & 1, wc, 19)) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const int t = q0 + row;
      uint16_t* dst = out + (static_cast<size_t>(b) * T + t) * out_stride + h * HD;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + lane_off + half * 32, o);
        tmem_ld_wait();
        if (t < T) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + half * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float* f = reinterpret_cast<const float*>(o) + q * 8;
            d4[q] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l), pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                               pack_bf16x2(f[4] * inv_l, f[5] * inv_l), pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

namespace wenc_host {

cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int q_col0,
                             int k_col0, int v_col0, uint16_t* out, int out_stride, int B, int T, int H,
                             uint32_t* err, cudaStream_t stream) {
  if (B <= 0 || T <= 0 || H <= 0) return cudaSuccess;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  dim3 grid((T + BQ - 1) / BQ, H, B);
  attn_fwd_kernel<<<grid, kThreads, SMEM, stream>>>(tq, tk, tv, q_col0, k_col0, v_col0, out, out_stride, T, scale_log2,
                                                     err);
  return cudaGetLastError();
}

}  // namespace wenc_host
