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
// How (sm_103a). A persistent kernel, one CTA per SM, walks work items of (256 queries, head,
// window), loading the next item's Q (double-buffered) and first K/V tiles and computing its
// first scores under the current item's last tiles and output. An item is two 128-row query
// tiles A and B that share every K and V tile, so the tensor pipe sees twice the work per K/V
// load and two softmax warps per SM sub-partition hide each other's latency:
//  - warp 0 streams Q_A, Q_B and K, V tiles of 64 keys (TMA, 128-byte swizzle; an fp32 head
//    row of 64 elements is two 128-byte swizzle columns);
//  - warp 2 transposes each V tile in shared memory into a [hd][key] K-major tile, so the PV
//    product reads a K-major B operand (V as loaded has hd, not keys, contiguous);
//  - one thread of warp 1 issues S_A = Q_A K_j^T and S_B = Q_B K_j^T (M128 N64, eight K=8 steps
//    each, both operands in shared memory) into double-buffered TMEM score tiles; one thread of
//    warp 3 issues O_A += P_A Vt_j and O_B += P_B Vt_j with P read from TMEM;
//  - warps 4-7 (tile A) and 8-11 (tile B) own one query row per thread: they read the row's 64
//    scores from TMEM, keep the running maximum and denominator (the online-softmax recurrence
//    of VANILLA_ATTN, base 2 with hd^-0.5 log2(e) folded in, maximum raised only when it grows
//    by more than 2^8), and write P, rounded to TF32, back over the same TMEM columns; O is
//    rescaled in TMEM when the maximum moved, after the previous product has completed.
// P never touches shared memory, and a score buffer is refilled once the product that read P
// from it has completed. Every barrier that a role waits on without waiting for each of its
// phases in turn exists once per buffer, so each parity wait is at most one phase from its
// target. (Twelve warps leave a thread 168 registers, thirteen only 128. Running the
// transpose in the producer warp to free a warp for a third issuer was slower.)
#include <math_constants.h>

#include <atomic>

#include "launch.h"
#include "ptx.cuh"

namespace {

using namespace wenc_dev;

constexpr int BQ = wenc_host::kAttnTf32BQ;    // query rows per tile (two tiles per CTA)
constexpr int BKV = wenc_host::kAttnTf32BKV;  // keys per tile
constexpr int HD = 64;
constexpr int NK = 2;     // K ring depth
constexpr int NVS = 2;    // V staging ring depth (as loaded: [key][hd])
constexpr int NVT = 2;    // transposed V ring depth ([hd][key])
constexpr int kSoftmaxWarp0 = 4;
constexpr int kThreads = 32 * (kSoftmaxWarp0 + 8);  // 4 control warps + two softmax warpgroups

constexpr uint32_t COL = 128;                        // bytes of one swizzled row (32 fp32)
constexpr uint32_t Q_CHUNK = BQ * COL;               // 16 KB: 128 rows x 32 hd
constexpr uint32_t Q_BYTES = 2 * Q_CHUNK;            // 32 KB per query tile
constexpr uint32_t KV_CHUNK = BKV * COL;             // 8 KB: 64 keys x 32 hd (or 64 hd x 32 keys)
constexpr uint32_t KV_BYTES = 2 * KV_CHUNK;          // 16 KB
constexpr uint32_t OFF_Q = 0;                        // two buffers of (Q_A, Q_B): this item's and the next's
constexpr uint32_t OFF_K = OFF_Q + 4 * Q_BYTES;
constexpr uint32_t OFF_VS = OFF_K + NK * KV_BYTES;
constexpr uint32_t OFF_VT = OFF_VS + NVS * KV_BYTES;
constexpr uint32_t OFF_BARS = OFF_VT + NVT * KV_BYTES;
// bars: q_full[2], q_empty[2]; k_full[NK], k_empty[NK]; vs_full[NVS], vs_empty[NVS]; vt_full[NVT],
// vt_empty[NVT]; per query tile t and buffer: s_full[t][2], s_free[t][2], p_full[t][2]; drain
constexpr int NUM_BARS = 4 + 2 * NK + 2 * NVS + 2 * NVT + 12 + 1;
constexpr size_t SMEM = 1024 + OFF_BARS + NUM_BARS * 8 + 16;
static_assert(SMEM <= 232448, "shared memory of the TF32 attention kernel");
// TMEM columns: S_A 0..127 (two buffers of 64), S_B 128..255, O_A 256..319, O_B 320..383
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T (kind::tf32, A = 128 lanes x 8 fp32 columns from a_tmem).
__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Byte offset of element (row, col) of a tile stored as 32-column chunks of 128-byte-swizzled
// rows: chunk col/32 at chunk_bytes * (col/32), 16-byte granule (col%32)/4 XOR (row%8).
__device__ __forceinline__ uint32_t sw_off(int row, int col, uint32_t chunk_bytes) {
  return (col >> 5) * chunk_bytes + row * COL + ((((col & 31) >> 2) ^ (row & 7)) << 4) + (col & 3) * 4;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tf32_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, int q_col0, int k_col0, int v_col0,
                     float* __restrict__ out, int out_stride, int T, int H, int n_items, float scale_log2,
                     uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ = s0 + OFF_Q, sK = s0 + OFF_K, sVS = s0 + OFF_VS, sVT = s0 + OFF_VT;
  const uint32_t bar0 = s0 + OFF_BARS;
  uint32_t nb = 0;
  const uint32_t q_full0 = bar0 + 8u * nb; nb += 2;   // [Q buffer]
  const uint32_t q_empty0 = bar0 + 8u * nb; nb += 2;  // [Q buffer]
  const uint32_t k_full0 = bar0 + 8u * nb; nb += NK;
  const uint32_t k_empty0 = bar0 + 8u * nb; nb += NK;
  const uint32_t vs_full0 = bar0 + 8u * nb; nb += NVS;
  const uint32_t vs_empty0 = bar0 + 8u * nb; nb += NVS;
  const uint32_t vt_full0 = bar0 + 8u * nb; nb += NVT;
  const uint32_t vt_empty0 = bar0 + 8u * nb; nb += NVT;
  const uint32_t s_full0 = bar0 + 8u * nb; nb += 4;   // [tile][buffer]
  const uint32_t s_free0 = bar0 + 8u * nb; nb += 4;   // [tile][buffer]
  const uint32_t p_full0 = bar0 + 8u * nb; nb += 4;   // [tile][buffer]
  const uint32_t drain = bar0 + 8u * nb;
  auto at = [](uint32_t base, int i) { return base + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BARS + NUM_BARS * 8);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, err};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_kv = (T + BKV - 1) / BKV;
  // Work item w (this CTA takes w = blockIdx.x, blockIdx.x + gridDim.x, ...): 256 queries of one
  // (window, head); w = (b * H + h) * n_qp + query-pair index. Every role walks the same items
  // and counts key tiles across them, so ring slots and barrier parities continue from one item
  // to the next.
  const int n_qp = (T + 2 * BQ - 1) / (2 * BQ);
  auto item_q0 = [&](int w) { return (w % n_qp) * 2 * BQ; };
  auto item_h = [&](int w) { return (w / n_qp) % H; };
  auto item_b = [&](int w) { return (w / n_qp) / H; };

  if (threadIdx.x == 0) {
    for (int u = 0; u < 2; ++u) {
      mbar_init(at(q_full0, u), 1);
      mbar_init(at(q_empty0, u), 1);  // the S issuer's commit after an item's last scores
    }
    for (int s = 0; s < NK; ++s) { mbar_init(at(k_full0, s), 1); mbar_init(at(k_empty0, s), 1); }
    for (int s = 0; s < NVS; ++s) { mbar_init(at(vs_full0, s), 1); mbar_init(at(vs_empty0, s), 1); }
    for (int s = 0; s < NVT; ++s) {
      mbar_init(at(vt_full0, s), 1);
      mbar_init(at(vt_empty0, s), 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(at(s_full0, i), 1);
      mbar_init(at(s_free0, i), 1);  // the PV product that read P from this buffer
      mbar_init(at(p_full0, i), 4);  // one arrival per softmax warp of the tile
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
  auto tS = [&](int t, int buf) { return tmem_base + 128u * t + 64u * buf; };
  auto tO = [&](int t) { return tmem_base + 256u + 64u * t; };

  // V transpose (warp 2, tile j): [key][hd] (as loaded) -> [hd][key], both 128-byte swizzled.
  // Lane l moves eight 4 x 4 blocks (4 keys x 4 hd columns) per tile: block (kq, dq) with
  // kq = ((l%8 + it) % 8) + 8 ((l/8) % 2), dq = l%8 + 8 (l/16), it = 0..7. Within each group
  // of eight lanes both the loads (row 4kq+e, granule dq%8 ^ row%8) and the stores (row
  // 4dq+i, granule kq%8 ^ row%8) hit eight distinct 16-byte granules: no bank conflicts.
  auto transpose_v = [&](int j) -> bool {
    const int lam = lane & 7, grp = lane >> 3;
    const int vs = j % NVS, vt = j % NVT;
    if (!mbar_wait_warp(at(vs_full0, vs), (j / NVS) & 1, wc, 38)) return false;
    if (!mbar_wait_warp(at(vt_empty0, vt), ((j / NVT) & 1) ^ 1u, wc, 39)) return false;
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
    return true;
  };


  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer, per item: Q_A, Q_B into the item's Q buffer (free once the
    // scores of the item two back are done), then K[j], V[j] for every key tile j; the next
    // item's Q and first tiles load while this item's last tiles run.
    int kc = 0, qi = 0;            // key tiles and items processed
    int k_issued = 0, v_issued = 0;  // K and V tiles whose copies were issued
    bool ok = true;
    for (int w = blockIdx.x, i = 0; ok && w < n_items; w += gridDim.x, ++i) {
      const int q0 = item_q0(w), h = item_h(w), b = item_b(w);
      const int qb = i & 1;
      if (!mbar_wait(at(q_empty0, qb), ((i >> 1) & 1) ^ 1u, wc, 30)) break;
      mbar_arrive_expect_tx(at(q_full0, qb), 2 * Q_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sQ + (2 * qb + t) * Q_BYTES + c * Q_CHUNK, &tq, at(q_full0, qb), q_col0 + h * HD + 32 * c,
                      q0 + t * BQ, b);
      qi = i + 1;
      for (int j = 0; j < n_kv; ++j, ++kc) {
        const int ks = kc % NK, vs = kc % NVS;
        if (!mbar_wait(at(k_empty0, ks), ((kc / NK) & 1) ^ 1u, wc, 31)) { ok = false; break; }
        mbar_arrive_expect_tx(at(k_full0, ks), KV_BYTES);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sK + ks * KV_BYTES + c * KV_CHUNK, &tk, at(k_full0, ks), k_col0 + h * HD + 32 * c, j * BKV, b);
        k_issued = kc + 1;
        if (!mbar_wait(at(vs_empty0, vs), ((kc / NVS) & 1) ^ 1u, wc, 32)) { ok = false; break; }
        mbar_arrive_expect_tx(at(vs_full0, vs), KV_BYTES);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sVS + vs * KV_BYTES + c * KV_CHUNK, &tv, at(vs_full0, vs), v_col0 + h * HD + 32 * c, j * BKV, b);
        v_issued = kc + 1;
      }
    }
    if (*abort_flag) {
      // Error path: let the copies already issued land before the CTA exits.
      for (int u = (qi > 2 ? qi - 2 : 0); u < qi; ++u) mbar_wait_drain(at(q_full0, u & 1), (u >> 1) & 1);
      for (int j = (k_issued > NK ? k_issued - NK : 0); j < k_issued; ++j)
        mbar_wait_drain(at(k_full0, j % NK), (j / NK) & 1);
      for (int j = (v_issued > NVS ? v_issued - NVS : 0); j < v_issued; ++j)
        mbar_wait_drain(at(vs_full0, j % NVS), (j / NVS) & 1);
    }
  } else if (warp == 2) {
    const int my_items = blockIdx.x < n_items ? (n_items - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1 : 0;
    for (int j = 0; j < my_items * n_kv; ++j)
      if (!transpose_v(j)) break;
  } else if ((warp == 1 || warp == 3) && lane == 0) {
    // ---------------- UMMA issuers (warp 1: scores of both tiles; warp 3: P V of both tiles).
    // A K step of 8 TF32 elements is 32 bytes inside a 128-byte swizzle row (+2 in the shared
    // memory descriptor's address field; steps 4..7 are in the second 32-column chunk), or 8
    // columns of the P tile in TMEM.
    constexpr uint32_t idesc = idesc_tf32_f32(BQ, 64);
    bool ok = true;
    if (warp == 1) {
      int g = 0;  // key tiles processed, across items
      for (int w = blockIdx.x, i = 0; ok && w < n_items; w += gridDim.x, ++i) {
        const int qb = i & 1;
        if (!mbar_wait(at(q_full0, qb), (i >> 1) & 1, wc, 33)) break;
        for (int j = 0; ok && j < n_kv; ++j, ++g) {
          const int ks = g % NK, buf = g & 1;
          if (!mbar_wait(at(k_full0, ks), (g / NK) & 1, wc, 34)) { ok = false; break; }
          for (int t = 0; t < 2 && ok; ++t) {
            if (g >= 2 && !mbar_wait(at(s_free0, 2 * t + buf), ((g - 2) >> 1) & 1, wc, 35)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < HD / 8; ++k) {
              const uint64_t qd =
                  sdesc_sw128(sQ + (2 * qb + t) * Q_BYTES + (k >> 2) * Q_CHUNK + (k & 3) * 32, 16, 1024);
              const uint64_t kd = sdesc_sw128(sK + ks * KV_BYTES + (k >> 2) * KV_CHUNK + (k & 3) * 32, 16, 1024);
              umma_tf32_ss(tS(t, buf), qd, kd, idesc, k > 0 ? 1u : 0u);
            }
            umma_commit(at(s_full0, 2 * t + buf));
          }
          if (ok) umma_commit(at(k_empty0, ks));
        }
        if (ok) umma_commit(at(q_empty0, qb));  // the item's Q buffer is free once its scores are done
      }
    } else {
      int g = 0;
      for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
        for (int j = 0; ok && j < n_kv; ++j, ++g) {
          const int vt = g % NVT;
          if (!mbar_wait(at(vt_full0, vt), (g / NVT) & 1, wc, 36)) { ok = false; break; }
          for (int t = 0; t < 2 && ok; ++t) {
            if (!mbar_wait(at(p_full0, 2 * t + (g & 1)), (g >> 1) & 1, wc, 37)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < BKV / 8; ++k) {
              const uint64_t vd = sdesc_sw128(sVT + vt * KV_BYTES + (k >> 2) * KV_CHUNK + (k & 3) * 32, 16, 1024);
              umma_tf32_ts(tO(t), tS(t, g & 1) + 8 * k, vd, idesc, (j > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(at(s_free0, 2 * t + (g & 1)));  // PV_t done: P buffer g%2 free, O updated
          }
          if (ok) umma_commit(at(vt_empty0, vt));
        }
      }
    }
    // Every MMA this thread issued completes before TMEM is released.
    umma_commit(drain);
    mbar_wait_drain(drain, 0);
  } else if (warp >= kSoftmaxWarp0) {
    // ---------------- softmax / correction / output: one query row per thread
    const int t = (warp - kSoftmaxWarp0) >> 2;  // query tile of this warpgroup
    const int quad = warp & 3;                   // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    int g = 0;  // key tiles processed, across items
    for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
      float m = -CUDART_INF_F;  // running maximum, in units of scale_log2
      float l = 0.0f;           // running denominator (sum of the TF32-rounded probabilities)
      for (int j = 0; j < n_kv; ++j, ++g) {
        const int buf = g & 1;
        if (!mbar_wait_warp(at(s_full0, 2 * t + buf), (g >> 1) & 1, wc, 40)) { ok = false; break; }
        tc_fence_after();
        float sv[BKV];
        {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(tS(t, buf) + lane_off, r0);
          tmem_ld_32x32b_x32(tS(t, buf) + lane_off + 32, r1);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            sv[e] = __uint_as_float(r0[e]);
            sv[32 + e] = __uint_as_float(r1[e]);
          }
        }

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

        // p = 2^(s * scale_log2 - m_new) rounded to TF32, in place, with packed fp32x2 arithmetic
        const uint64_t c2 = pack_f32x2(scale_log2, scale_log2);
        const uint64_t nm2 = pack_f32x2(-m_new, -m_new);
        uint64_t sum2a = pack_f32x2(0.0f, 0.0f), sum2b = sum2a;
#pragma unroll
        for (int i = 0; i < BKV / 2; ++i) {
          float a0, a1;
          unpack_f32x2(fma_f32x2(pack_f32x2(sv[2 * i], sv[2 * i + 1]), c2, nm2), a0, a1);
          sv[2 * i] = round_tf32(ex2_approx(a0));
          sv[2 * i + 1] = round_tf32(ex2_approx(a1));
          if (i & 1) sum2b = add_f32x2(sum2b, pack_f32x2(sv[2 * i], sv[2 * i + 1]));
          else sum2a = add_f32x2(sum2a, pack_f32x2(sv[2 * i], sv[2 * i + 1]));
        }
        float sa0, sa1, sb0, sb1;
        unpack_f32x2(sum2a, sa0, sa1);
        unpack_f32x2(sum2b, sb0, sb1);
        const float sum = (sa0 + sa1) + (sb0 + sb1);

        {
          // P over this tile's scores in TMEM (the PV product reads its A operand from there)
          uint32_t p0[32], p1[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            p0[e] = __float_as_uint(sv[e]);
            p1[e] = __float_as_uint(sv[32 + e]);
          }
          tmem_st_32x32b_x32(tS(t, buf) + lane_off, p0);
          tmem_st_32x32b_x32(tS(t, buf) + lane_off + 32, p1);
        }
        if (j > 0 && __any_sync(0xffffffffu, m_new != m)) {
          // O holds the products of tiles 0..j-1 once PV[j-1] is complete; rescale it.
          if (!mbar_wait_warp(at(s_free0, 2 * t + ((g - 1) & 1)), ((g - 1) >> 1) & 1, wc, 41)) { ok = false; break; }
          tc_fence_after();
          {
            uint32_t o0[32], o1[32];
            tmem_ld_32x32b_x32(tO(t) + lane_off, o0);
            tmem_ld_32x32b_x32(tO(t) + lane_off + 32, o1);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              o0[c] = __float_as_uint(__uint_as_float(o0[c]) * alpha);
              o1[c] = __float_as_uint(__uint_as_float(o1[c]) * alpha);
            }
            tmem_st_32x32b_x32(tO(t) + lane_off, o0);
            tmem_st_32x32b_x32(tO(t) + lane_off + 32, o1);
          }
        }
        tmem_st_wait();  // P (and a rescaled O) are in TMEM before the product is released
        l = l * alpha + sum;
        m = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(at(p_full0, 2 * t + buf));
      }
      // The item's last PV_t complete (it completes after the one before; per-buffer barriers
      // keep each parity wait within one phase of its target: the PV_t two back is known
      // complete here). The next item's first PV_t, which overwrites O, waits for P that this
      // warp writes only after the reads below.
      if (!ok || !mbar_wait_warp(at(s_free0, 2 * t + ((g - 1) & 1)), ((g - 1) >> 1) & 1, wc, 43)) break;
      {
        tc_fence_after();
        const int tq_row = item_q0(w) + t * BQ + row;
        const int b = item_b(w), h = item_h(w);
        const float inv_l = 1.0f / l;
        float* dst = out + (static_cast<size_t>(b) * T + tq_row) * out_stride + h * HD;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO(t) + lane_off + half * 32, o);
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
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Shared-memory opt-in, once per device (a repeat by a racing host thread is harmless).
  static std::atomic<int> configured_device{-1};
  if (configured_device.load(std::memory_order_acquire) != dev) {
    e = cudaFuncSetAttribute(attn_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
    if (e != cudaSuccess) return e;
    configured_device.store(dev, std::memory_order_release);
  }
  int num_sms = 0;
  e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  const long long items = static_cast<long long>((T + 2 * BQ - 1) / (2 * BQ)) * H * B;
  if (items > (1LL << 30)) return cudaErrorInvalidValue;
  // Persistent: one CTA per SM, each walking the items w = blockIdx.x + k * gridDim.x.
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  return launch_pdl(attn_tf32_kernel, dim3(grid), dim3(kThreads), SMEM, stream, tq, tk, tv, q_col0, k_col0, v_col0,
                    out, out_stride, T, H, static_cast<int>(items), scale_log2, err);
}

}  // namespace wenc_host
