// attn_tf32.cu -- the block's attention with TF32 operands and fp32 activations.
//
// Same computation as attn.cu (inferencelayer 0.2.4 src/whisper_gpu.rs, VANILLA_ATTN;
// turbospark-runtime 0.3.0 src/whisper/metal.rs, encode_layer): per window b, head h and query
// row i, s_j = (q_i . k_j) * hd^-0.5 over all T keys, p = softmax(s), o_i = sum_j p_j v_j.
// Q, K, V and the output are fp32 [B, T, row]; the products run as kind::tf32 MMAs (fp32
// operands read as TF32, fp32 accumulation), the probabilities are rounded to TF32 before the
// PV product and the output is written as fp32 rounded to TF32 (the operand of the TF32
// out-projection GEMM that follows it).
//
// How (sm_103a). One CTA per (128 queries, head, window):
//  - warp 0 streams Q once and K, V tiles of 64 keys (TMA, 128-byte swizzle; an fp32 head row
//    of 64 elements is two 128-byte swizzle columns);
//  - warp 2 transposes each V tile in shared memory into a [hd][key] K-major tile, so both
//    products read K-major operands: S = Q K^T contracts over hd, O += P V^T-as-B contracts over
//    keys, and V as loaded has hd, not keys, contiguous;
//  - one thread of warp 1 issues S_j = Q K_j^T (M128 N64, eight K=8 steps) into one of two TMEM
//    score buffers; one thread of warp 3 issues O += P_j Vt_j (M128 N64) into the TMEM
//    accumulator;
//  - warps 4-7 own one query row per thread: they read the row's 64 scores from TMEM, keep the
//    running maximum and denominator (the online-softmax recurrence of VANILLA_ATTN, base 2 with
//    hd^-0.5 log2(e) folded in, maximum raised only when it grows by more than 2^8), write P
//    rounded to TF32 into swizzled shared memory and rescale O in TMEM when the maximum moves.
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"

namespace {

using namespace wenc_dev;

constexpr int BQ = wenc_host::kAttnTf32BQ;  // query rows per CTA
constexpr int BKV = wenc_host::kAttnTf32BKV;  // keys per tile
constexpr int HD = 64;
constexpr int NK = 3;     // K ring depth
constexpr int NVS = 2;    // V staging ring depth (as loaded: [key][hd])
constexpr int NVT = 2;    // transposed V ring depth ([hd][key])
constexpr int kThreads = 256;

constexpr uint32_t COL = 128;                        // bytes of one swizzled row (32 fp32)
constexpr uint32_t Q_CHUNK = BQ * COL;               // 16 KB: 128 rows x 32 hd
constexpr uint32_t Q_BYTES = 2 * Q_CHUNK;
constexpr uint32_t KV_CHUNK = BKV * COL;             // 8 KB: 64 keys x 32 hd (or 64 hd x 32 keys)
constexpr uint32_t KV_BYTES = 2 * KV_CHUNK;          // 16 KB
constexpr uint32_t P_CHUNK = BQ * COL;               // 16 KB: 128 rows x 32 keys
constexpr uint32_t P_BYTES = 2 * P_CHUNK;            // 32 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_VS = OFF_K + NK * KV_BYTES;
constexpr uint32_t OFF_VT = OFF_VS + NVS * KV_BYTES;
constexpr uint32_t OFF_P = OFF_VT + NVT * KV_BYTES;
constexpr uint32_t OFF_BARS = OFF_P + 2 * P_BYTES;
// bars: q_full; k_full[NK], k_empty[NK]; vs_full[NVS], vs_empty[NVS]; vt_full[NVT], vt_empty[NVT];
// s_full[2], s_free[2]; p_full[2]; pv_done[2]; drain
constexpr int NUM_BARS = 1 + 2 * NK + 2 * NVS + 2 * NVT + 8 + 1;
constexpr size_t SMEM = 1024 + OFF_BARS + NUM_BARS * 8 + 16;
static_assert(SMEM <= 232448, "shared memory of the TF32 attention kernel");
constexpr uint32_t TMEM_COLS = 256;  // S0 0..63, S1 64..127, O 128..191
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Byte offset of element (row, col) of a tile stored as 32-column chunks of 128-byte-swizzled
// rows: chunk col/32 at chunk_bytes * (col/32), 16-byte granule (col%32)/4 XOR (row%8).
__device__ __forceinline__ uint32_t sw_off(int row, int col, uint32_t chunk_bytes) {
  return (col >> 5) * chunk_bytes + row * COL + ((((col & 31) >> 2) ^ (row & 7)) << 4) + (col & 3) * 4;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tf32_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, int q_col0, int k_col0, int v_col0,
                     float* __restrict__ out, int out_stride, int T, float scale_log2, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ = s0 + OFF_Q, sK = s0 + OFF_K, sVS = s0 + OFF_VS, sVT = s0 + OFF_VT, sP = s0 + OFF_P;
  const uint32_t bar0 = s0 + OFF_BARS;
  uint32_t nb = 0;
  const uint32_t q_full = bar0 + 8u * nb++;
  const uint32_t k_full0 = bar0 + 8u * nb; nb += NK;
  const uint32_t k_empty0 = bar0 + 8u * nb; nb += NK;
  const uint32_t vs_full0 = bar0 + 8u * nb; nb += NVS;
  const uint32_t vs_empty0 = bar0 + 8u * nb; nb += NVS;
  const uint32_t vt_full0 = bar0 + 8u * nb; nb += NVT;
  const uint32_t vt_empty0 = bar0 + 8u * nb; nb += NVT;
  const uint32_t s_full0 = bar0 + 8u * nb; nb += 2;
  const uint32_t s_free0 = bar0 + 8u * nb; nb += 2;
  const uint32_t p_full0 = bar0 + 8u * nb; nb += 2;
  const uint32_t pv_done0 = bar0 + 8u * nb; nb += 2;
  const uint32_t drain = bar0 + 8u * nb;
  auto at = [](uint32_t base, int i) { return base + 8u * i; };
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
    for (int s = 0; s < NK; ++s) { mbar_init(at(k_full0, s), 1); mbar_init(at(k_empty0, s), 1); }
    for (int s = 0; s < NVS; ++s) { mbar_init(at(vs_full0, s), 1); mbar_init(at(vs_empty0, s), 1); }
    for (int s = 0; s < NVT; ++s) { mbar_init(at(vt_full0, s), 1); mbar_init(at(vt_empty0, s), 1); }
    for (int t = 0; t < 2; ++t) {
      mbar_init(at(s_full0, t), 1);
      mbar_init(at(s_free0, t), 4);   // one arrival per softmax warp
      mbar_init(at(p_full0, t), 4);
      mbar_init(at(pv_done0, t), 1);
    }
    mbar_init(drain, 2);  // one commit per MMA-issuing thread
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
  pdl_trigger();  // TMEM is held: the next kernel may be scheduled
  pdl_wait();     // Q, K, V from the previous kernel are complete from here on
  const uint32_t tO = tmem_base + 128u;
  auto tS = [&](int buf) { return tmem_base + 64u * buf; };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: Q; then K[j], V[j] for every key tile j
    mbar_arrive_expect_tx(q_full, Q_BYTES);
    for (int c = 0; c < 2; ++c) tma_load_3d(sQ + c * Q_CHUNK, &tq, q_full, q_col0 + h * HD + 32 * c, q0, b);
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int ks = j % NK, vs = j % NVS;
      if (!mbar_wait(at(k_empty0, ks), ((j / NK) & 1) ^ 1u, wc, 31)) { ok = false; break; }
      mbar_arrive_expect_tx(at(k_full0, ks), KV_BYTES);
      for (int c = 0; c < 2; ++c)
        tma_load_3d(sK + ks * KV_BYTES + c * KV_CHUNK, &tk, at(k_full0, ks), k_col0 + h * HD + 32 * c, j * BKV, b);
      k_issued = j + 1;
      if (!mbar_wait(at(vs_empty0, vs), ((j / NVS) & 1) ^ 1u, wc, 32)) { ok = false; break; }
      mbar_arrive_expect_tx(at(vs_full0, vs), KV_BYTES);
      for (int c = 0; c < 2; ++c)
        tma_load_3d(sVS + vs * KV_BYTES + c * KV_CHUNK, &tv, at(vs_full0, vs), v_col0 + h * HD + 32 * c, j * BKV, b);
      v_issued = j + 1;
    }
    if (*abort_flag) {
      // Error path: let the copies already issued land before the CTA exits.
      mbar_wait_drain(q_full, 0);
      for (int j = (k_issued > NK ? k_issued - NK : 0); j < k_issued; ++j) mbar_wait_drain(at(k_full0, j % NK), (j / NK) & 1);
      for (int j = (v_issued > NVS ? v_issued - NVS : 0); j < v_issued; ++j)
        mbar_wait_drain(at(vs_full0, j % NVS), (j / NVS) & 1);
    }
  } else if ((warp == 1 || warp == 3) && lane == 0) {
    // ---------------- UMMA issuers (warp 1: scores; warp 3: P V). A K step of 8 TF32 elements
    // is 32 bytes inside a 128-byte swizzle row (+2 in the descriptor's address field); steps
    // 4..7 are in the second 32-column chunk of the operand.
    constexpr uint32_t idesc = idesc_tf32_f32(BQ, 64);
    bool ok = true;
    if (warp == 1) {
      ok = mbar_wait(q_full, 0, wc, 33);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int ks = j % NK, buf = j & 1;
        if (!mbar_wait(at(k_full0, ks), (j / NK) & 1, wc, 34)) break;
        if (j >= 2 && !mbar_wait(at(s_free0, buf), ((j - 2) >> 1) & 1, wc, 35)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < HD / 8; ++k) {
          const uint64_t qd = sdesc_sw128(sQ + (k >> 2) * Q_CHUNK + (k & 3) * 32, 16, 1024);
          const uint64_t kd = sdesc_sw128(sK + ks * KV_BYTES + (k >> 2) * KV_CHUNK + (k & 3) * 32, 16, 1024);
          umma_tf32_ss(tS(buf), qd, kd, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(at(s_full0, buf));
        umma_commit(at(k_empty0, ks));
      }
    } else {
      for (int j = 0; ok && j < n_kv; ++j) {
        const int vt = j % NVT, buf = j & 1;
        if (!mbar_wait(at(p_full0, buf), (j >> 1) & 1, wc, 36)) break;
        if (!mbar_wait(at(vt_full0, vt), (j / NVT) & 1, wc, 37)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BKV / 8; ++k) {
          const uint64_t pd = sdesc_sw128(sP + buf * P_BYTES + (k >> 2) * P_CHUNK + (k & 3) * 32, 16, 1024);
          const uint64_t vd = sdesc_sw128(sVT + vt * KV_BYTES + (k >> 2) * KV_CHUNK + (k & 3) * 32, 16, 1024);
          umma_tf32_ss(tO, pd, vd, idesc, (j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(at(pv_done0, buf));
        umma_commit(at(vt_empty0, vt));
      }
    }
    // Every MMA this thread issued completes before TMEM is released.
    umma_commit(drain);
    mbar_wait_drain(drain, 0);
  } else if (warp == 2) {
    // ---------------- V transpose: [key][hd] (as loaded) -> [hd][key], both 128-byte swizzled.
    // Lane l moves eight 4 x 4 blocks (4 keys x 4 hd columns) per tile: block (kq, dq) with
    // kq = ((l%8 + it) % 8) + 8 ((l/8) % 2), dq = l%8 + 8 (l/16), it = 0..7. Within each group
    // of eight lanes both the loads (row 4kq+e, granule dq%8 ^ row%8) and the stores (row
    // 4dq+i, granule kq%8 ^ row%8) hit eight distinct 16-byte granules: no bank conflicts.
    const int lam = lane & 7, grp = lane >> 3;
    for (int j = 0; j < n_kv; ++j) {
      const int vs = j % NVS, vt = j % NVT;
      if (!mbar_wait_warp(at(vs_full0, vs), (j / NVS) & 1, wc, 38)) break;
      if (!mbar_wait_warp(at(vt_empty0, vt), ((j / NVT) & 1) ^ 1u, wc, 39)) break;
      const uint32_t src = sVS + vs * KV_BYTES, dst = sVT + vt * KV_BYTES;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int kq = ((lam + it) & 7) + 8 * (grp & 1);
        const int dq = lam + 8 * (grp >> 1);
        float4 r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = lds_f4(src + sw_off(4 * kq + e, 4 * dq, KV_CHUNK));
        sts_f4(dst + sw_off(4 * dq + 0, 4 * kq, KV_CHUNK), r[0].x, r[1].x, r[2].x, r[3].x);
        sts_f4(dst + sw_off(4 * dq + 1, 4 * kq, KV_CHUNK), r[0].y, r[1].y, r[2].y, r[3].y);
        sts_f4(dst + sw_off(4 * dq + 2, 4 * kq, KV_CHUNK), r[0].z, r[1].z, r[2].z, r[3].z);
        sts_f4(dst + sw_off(4 * dq + 3, 4 * kq, KV_CHUNK), r[0].w, r[1].w, r[2].w, r[3].w);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(at(vs_empty0, vs));
        mbar_arrive(at(vt_full0, vt));
      }
    }
  } else if (warp >= 4) {
    // ---------------- softmax / correction / output: one query row per thread
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float m = -CUDART_INF_F;  // running maximum, in units of scale_log2
    float l = 0.0f;           // running denominator (sum of the TF32-rounded probabilities)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int buf = j & 1;
      if (!mbar_wait_warp(at(s_full0, buf), (j >> 1) & 1, wc, 40)) { ok = false; break; }
      tc_fence_after();
      float sv[BKV];
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tS(buf) + lane_off + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) sv[c * 32 + e] = __uint_as_float(r[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(at(s_free0, buf));  // the MMA may overwrite this score buffer

      const int valid = T - j * BKV;  // keys of this tile inside the window
      if (valid < BKV) {              // only the last tile can be partial (warp-uniform)
#pragma unroll
        for (int c = 0; c < BKV; ++c) sv[c] = (c < valid) ? sv[c] : -CUDART_INF_F;
      }
      float mc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a = fmax3(sv[16 * k], sv[16 * k + 1], sv[16 * k + 2]);
#pragma unroll
        for (int e = 3; e < 15; e += 2) a = fmax3(a, sv[16 * k + e], sv[16 * k + e + 1]);
        mc[k] = fmaxf(a, sv[16 * k + 15]);
      }
      const float mx_s = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])) * scale_log2;
      const float m_new = (mx_s > m + kRescaleThreshold) ? mx_s : m;
      const float alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)

      // P buffer `buf` was last read by the product of tile j-2.
      if (j >= 2 && !mbar_wait_warp(at(pv_done0, buf), ((j - 2) >> 1) & 1, wc, 41)) { ok = false; break; }
      float sum = 0.0f;
      const uint32_t prow = sP + buf * P_BYTES;
#pragma unroll
      for (int c4 = 0; c4 < BKV / 4; ++c4) {
        const float p0 = round_tf32(ex2_approx(fmaf(sv[4 * c4 + 0], scale_log2, -m_new)));
        const float p1 = round_tf32(ex2_approx(fmaf(sv[4 * c4 + 1], scale_log2, -m_new)));
        const float p2 = round_tf32(ex2_approx(fmaf(sv[4 * c4 + 2], scale_log2, -m_new)));
        const float p3 = round_tf32(ex2_approx(fmaf(sv[4 * c4 + 3], scale_log2, -m_new)));
        sum += (p0 + p1) + (p2 + p3);
        sts_f4(prow + sw_off(row, 4 * c4, P_CHUNK), p0, p1, p2, p3);
      }
      if (j >= 1 && __any_sync(0xffffffffu, m_new != m)) {
        // O holds the products of tiles 0..j-1 once PV[j-1] is complete; rescale it.
        if (!mbar_wait_warp(at(pv_done0, (j - 1) & 1), ((j - 1) >> 1) & 1, wc, 42)) { ok = false; break; }
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
      }
      l = l * alpha + sum;
      m = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(at(p_full0, buf));
    }
    if (ok && mbar_wait_warp(at(pv_done0, (n_kv - 1) & 1), ((n_kv - 1) >> 1) & 1, wc, 43)) {
      tc_fence_after();
      const int tq_row = q0 + row;
      const float inv_l = 1.0f / l;
      float* dst = out + (static_cast<size_t>(b) * T + tq_row) * out_stride + h * HD;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + lane_off + half * 32, o);
        tmem_ld_wait();
        if (tq_row < T) {
          float4* d4 = reinterpret_cast<float4*>(dst + half * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d4[q] = make_float4(round_tf32(__uint_as_float(o[4 * q]) * inv_l), round_tf32(__uint_as_float(o[4 * q + 1]) * inv_l),
                                round_tf32(__uint_as_float(o[4 * q + 2]) * inv_l), round_tf32(__uint_as_float(o[4 * q + 3]) * inv_l));
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

cudaError_t launch_attention_tf32(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int q_col0,
                                  int k_col0, int v_col0, float* out, int out_stride, int B, int T, int H,
                                  uint32_t* err, cudaStream_t stream) {
  if (B <= 0 || T <= 0 || H <= 0) return cudaSuccess;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  dim3 grid((T + BQ - 1) / BQ, H, B);
  return launch_pdl(attn_tf32_kernel, grid, dim3(kThreads), SMEM, stream, tq, tk, tv, q_col0, k_col0, v_col0, out,
                    out_stride, T, scale_log2, err);
}

}  // namespace wenc_host
