// attn.cu -- non-causal scaled-dot attention of one encoder window, fused (flash style).
//
// What it computes (inferencelayer 0.2.4 src/whisper_gpu.rs, VANILLA_ATTN; turbospark-runtime
// 0.3.0 src/whisper/metal.rs, encode_layer): for every window b, head h and query row i,
//   s_j = (q_i . k_j) * hd^-0.5 over all T keys,  p = softmax(s),  o_i = sum_j p_j v_j.
// No mask beyond the window's own length, no positional term.
//
// How (sm_103a). A persistent kernel, one CTA per SM, walks work items of (256 queries, head,
// window); the next item's Q and first K/V tiles load, and its first scores are computed, while
// the current item's last tiles and output run (a CTA per item paid ~30% of the time in its
// ramp-up and drain). The 256 queries are two 128-row tiles A and B that share every K/V tile:
//  - warp 0 streams Q_A, Q_B (two buffers: this item's and the next's) and K, V tiles of 128
//    keys (TMA, 128-byte swizzle) through rings of their own, in the order the tensor pipe
//    consumes them;
//  - one thread of warp 1 issues S_A = Q_A K_j^T and S_B = Q_B K_j^T (M128 N128 K64, into TMEM)
//    as soon as the scores of tile j-1 have been read; one thread each of warps 2 and 3 issues
//    O_A += P_A V_j and O_B += P_B V_j (M128 N64, P from TMEM, V read MN-major from shared
//    memory, O accumulated in TMEM) once P of tile j is written (one issuing thread cannot keep
//    the tensor pipe fed with N = 64 MMAs);
//  - warps 4-7 (tile A) and 8-11 (tile B) own one query row per thread: they read the row's 128
//    scores from TMEM, keep the running maximum and denominator in registers (the online-softmax
//    recurrence of VANILLA_ATTN, in base 2 with hd^-0.5*log2(e) folded in), write P as bf16 pairs
//    into the tile's P columns of TMEM (the PV product reads its A operand from there: no P
//    traffic through shared memory) and rescale O in TMEM when the running maximum moves by more
//    than 2^8. The two tiles take turns on the exponentials (ping-pong), so one tile's exps run
//    while the other tile loads scores, stores P or waits, and the tensor pipe runs the other
//    tile's products meanwhile. The turn passes through hardware named barriers: a tile's warps
//    resume a few tens of cycles after the other tile's arrive, where an mbarrier wait took
//    ~115 (210 -> 197 us at T = 1500). No T x T score buffer exists.
// The control warpgroup (warps 0-3) hands registers to the softmax warpgroups at start-up
// (setmaxnreg: 104 and 200 per thread instead of 168 for all), which keeps a row's scores and the
// exponential pipeline in registers (211.6 -> 197.5 us at large-v3 dims, B = 16; the four score
// loads then share one wait: 195.6 us).
// Key tiles of 128 make the S products full-rate (N = 128); the PV products have N = hd = 64.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <atomic>

#include "launch.h"
#include "ptx.cuh"

namespace {

using namespace wenc_dev;

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 with bf16 operands; A = 128 lanes x 8 columns, each
// 32-bit column holding two consecutive K elements (the lower one in the low half).
// Hardware named barriers (ids 1 and 2; __syncthreads uses 0): `count` threads in whole warps.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

constexpr int BQ = wenc_host::kAttnBQ;    // query rows per tile (two tiles per CTA)
constexpr int BKV = wenc_host::kAttnBKV;  // keys per tile
constexpr int HD = 64;
constexpr int NK = 3;                     // K ring depth
constexpr int NV = 3;                     // V ring depth
constexpr int kThreads = 384;             // producer, 3 MMA issuers, 2 softmax warpgroups
// Registers per thread after the start-up reallocation (setmaxnreg): the control warpgroup
// (producer and MMA issuers) gives up registers that the two softmax warpgroups take, which keeps
// a row's 128 scores and the exponential pipeline out of local memory. The sum must fit in what
// the CTA is launched with (checked on the host before the first launch).
constexpr int kCtrlRegs = 104;
constexpr int kSoftmaxRegs = 200;
constexpr int kRegsNeeded = kCtrlRegs * 128 + kSoftmaxRegs * 256;
static_assert(kRegsNeeded <= (65536 / kThreads) / 8 * 8 * kThreads, "register split exceeds the launch budget");

constexpr uint32_t Q_BYTES = BQ * HD * 2;           // 16 KB per query tile
constexpr uint32_t KV_BYTES = BKV * HD * 2;         // 16 KB per K or V tile
constexpr uint32_t OFF_Q = 0;                       // two buffers of (Q_A, Q_B): this item's and the next's
constexpr uint32_t OFF_K = OFF_Q + 4 * Q_BYTES;
constexpr uint32_t OFF_V = OFF_K + NK * KV_BYTES;
constexpr uint32_t OFF_BARS = OFF_V + NV * KV_BYTES;
// bars: q_full[2], q_empty[2], k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], and per query
// tile t: s_full[t], s_free[t], p_full[t], pv_done[t]; drain. (The exponential turn uses the
// hardware named barriers 1 and 2.)
constexpr int NUM_BARS = 4 + 2 * NK + 2 * NV + 8 + 1;
constexpr size_t SMEM = 1024 + OFF_BARS + NUM_BARS * 8 + 16;
constexpr uint32_t TMEM_COLS = 512;  // S_A 0..127, S_B 128..255, O_A 256..319, O_B 320..383, P_A 384..447, P_B 448..511
// Grow the running maximum only when a tile's maximum exceeds it by more than this (log2
// units); otherwise keep it, so p <= 2^8 and O is rescaled rarely. The result is unchanged:
// numerator and denominator always use the same reference maximum.
constexpr float kRescaleThreshold = 8.0f;

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, int q_col0, int k_col0, int v_col0,
                    uint16_t* __restrict__ out, int out_stride, int T, int H, int n_items, float scale_log2,
                    int n_splits, int tiles_per_split, float* __restrict__ part_o, float2* __restrict__ part_ml,
                    uint32_t* err, int stop_after) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ = s0 + OFF_Q, sK = s0 + OFF_K, sV = s0 + OFF_V;
  const uint32_t bar0 = s0 + OFF_BARS;
  auto q_full = [&](int u) { return bar0 + 8u * u; };
  auto q_empty = [&](int u) { return bar0 + 8u * (2 + u); };
  auto k_full = [&](int s) { return bar0 + 8u * (4 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (4 + NK + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (4 + 2 * NK + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (4 + 2 * NK + NV + s); };
  const uint32_t tb0 = bar0 + 8u * (4 + 2 * NK + 2 * NV);
  auto s_full = [&](int t) { return tb0 + 8u * t; };
  auto s_free = [&](int t) { return tb0 + 16u + 8u * t; };
  auto p_full = [&](int t) { return tb0 + 32u + 8u * t; };
  auto pv_done = [&](int t) { return tb0 + 48u + 8u * t; };
  const uint32_t drain = tb0 + 64u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BARS + NUM_BARS * 8);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, err};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Work item w (this CTA takes w = blockIdx.x, blockIdx.x + gridDim.x, ...): 256 queries of one
  // (window, head) against one split of its keys. w = (b * H + h) * n_x + x with
  // x = query-pair index * n_splits + split; a split covers key tiles [kv0, kv0 + n_kv) of the
  // window (all of them when n_splits == 1).
  const int n_kv_all = (T + BKV - 1) / BKV;
  const int n_x = ((T + 2 * BQ - 1) / (2 * BQ)) * n_splits;
  const int n_windows = n_items / (n_x * H);
  struct Item {
    int q0, h, b, split, kv0, n_kv;
  };
  auto decode = [&](int w) {
    Item it;
    const int x = w % n_x, bh = w / n_x;
    it.h = bh % H;
    it.b = bh / H;
    it.split = x % n_splits;
    it.q0 = (x / n_splits) * 2 * BQ;
    it.kv0 = it.split * tiles_per_split;
    it.n_kv = min(tiles_per_split, n_kv_all - it.kv0);  // >= 1 by construction
    return it;
  };

  if (threadIdx.x == 0) {
    for (int u = 0; u < 2; ++u) {
      mbar_init(q_full(u), 1);
      mbar_init(q_empty(u), 1);  // released by the S issuer's commit after an item's last S
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 2);  // released by both PV issuers
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(s_free(t), 4);  // one arrival per softmax warp of the tile
      mbar_init(p_full(t), 4);
      mbar_init(pv_done(t), 1);
    }
    mbar_init(drain, 3);  // one commit per MMA-issuing thread
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
  auto tS = [&](int t) { return tmem_base + 128u * t; };
  auto tO = [&](int t) { return tmem_base + 256u + 64u * t; };
  auto tP = [&](int t) { return tmem_base + 384u + 64u * t; };  // P as bf16 pairs: 64 columns per tile

  // Every role walks the same items in the same order and counts K/V tiles across them (kc,
  // vc, g below), so ring slots and barrier parities continue from one item to the next.
  if (warp < 4) {
    // control warpgroup: registers to the softmax warpgroups first
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kCtrlRegs) : "memory");
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer, per item: Q_A, Q_B into the item's Q buffer (free once the
      // S products of the item two back are done), then K0, then (K[j], V[j-1]) for j >= 1, then
      // V[n-1]; the next item's Q and first K tiles load while this item's last tiles run.
      int kc = 0, vc = 0, qi = 0;  // K tiles, V tiles and items issued
      auto load_k = [&](const Item& it, int j) -> bool {
        if (stop_after >= 0 && kc >= stop_after) {
          // self-test: this producer gives up here as if a wait had run out (site 31)
          *abort_flag = 1u;
          *reinterpret_cast<volatile uint32_t*>(err) = kErrTimeout | (31u << 8);
          return false;
        }
        const int st = kc % NK;
        if (!mbar_wait(k_empty(st), ((kc / NK) & 1) ^ 1u, wc, 11)) return false;
        mbar_arrive_expect_tx(k_full(st), KV_BYTES);
        tma_load_3d(sK + st * KV_BYTES, &tk, k_full(st), k_col0 + it.h * HD, (it.kv0 + j) * BKV, it.b);
        ++kc;
        return true;
      };
      auto load_v = [&](const Item& it, int j) -> bool {
        const int st = vc % NV;
        if (!mbar_wait(v_empty(st), ((vc / NV) & 1) ^ 1u, wc, 10)) return false;
        mbar_arrive_expect_tx(v_full(st), KV_BYTES);
        tma_load_3d(sV + st * KV_BYTES, &tv, v_full(st), v_col0 + it.h * HD, (it.kv0 + j) * BKV, it.b);
        ++vc;
        return true;
      };
      bool ok = true;
      for (int w = blockIdx.x, i = 0; ok && w < n_items; w += gridDim.x, ++i) {
        const Item it = decode(w);
        const int qb = i & 1;
        if (!in_bounds(it.q0 >= 0 && it.q0 < T && it.h >= 0 && it.h < H && it.b >= 0 && it.b < n_windows &&
                           it.kv0 >= 0 && it.n_kv >= 1 && it.kv0 + it.n_kv <= n_kv_all && it.split < n_splits,
                       err, 72)) {
          *abort_flag = 1u;  // an item outside the problem: stop as a failed wait would
          break;
        }
        if (!mbar_wait(q_empty(qb), ((i >> 1) & 1) ^ 1u, wc, 9)) break;
        mbar_arrive_expect_tx(q_full(qb), 2 * Q_BYTES);
        tma_load_3d(sQ + qb * 2 * Q_BYTES, &tq, q_full(qb), q_col0 + it.h * HD, it.q0, it.b);
        tma_load_3d(sQ + qb * 2 * Q_BYTES + Q_BYTES, &tq, q_full(qb), q_col0 + it.h * HD, it.q0 + BQ, it.b);
        qi = i + 1;
        for (int j = 0; ok && j <= it.n_kv; ++j) {
          if (j < it.n_kv) ok = load_k(it, j);
          if (ok && j >= 1) ok = load_v(it, j - 1);
        }
      }
      if (*abort_flag) {
        // Error path: let the copies already issued land before the CTA exits.
        for (int u = (qi > 2 ? qi - 2 : 0); u < qi; ++u) mbar_wait_drain(q_full(u & 1), (u >> 1) & 1);
        for (int j = (kc > NK ? kc - NK : 0); j < kc; ++j) mbar_wait_drain(k_full(j % NK), (j / NK) & 1);
        for (int j = (vc > NV ? vc - NV : 0); j < vc; ++j) mbar_wait_drain(v_full(j % NV), (j / NV) & 1);
      }
    } else if (warp >= 1 && warp <= 3 && lane == 0) {
      // ---------------- UMMA issuers. A single thread cannot issue MMAs fast enough to keep the
      // tensor pipe busy with N = 64 products, so three threads share the work: warp 1 issues
      // S_A = Q_A K_j^T and S_B = Q_B K_j^T as soon as the scores of tile j-1 have been read;
      // warps 2 and 3 issue O_A += P_A V_j and O_B += P_B V_j once P of tile j is written.
      // Descriptors are built once per operand tile; a K step of 16 elements advances the start
      // address by 32 bytes (K-major, inside the 128-byte swizzle row: +2 in the >>4 field) or by
      // 16 rows of 128 bytes (the MN-major V tile: +128).
      bool ok = true;
      if (warp == 1) {
        constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV, false);  // B = K tile, K-major, N = 128
        int kc = 0;  // K tiles consumed, across items
        for (int w = blockIdx.x, i = 0; ok && w < n_items; w += gridDim.x, ++i) {
          const int n_kv = decode(w).n_kv;
          const int qb = i & 1;
          if (!mbar_wait(q_full(qb), (i >> 1) & 1, wc, 12)) break;
          for (int j = 0; ok && j < n_kv; ++j, ++kc) {
            const int st = kc % NK;
            if (!mbar_wait(k_full(st), (kc / NK) & 1, wc, 13)) { ok = false; break; }
            const uint64_t kdesc = sdesc_sw128(sK + st * KV_BYTES, 16, 1024);
            for (int t = 0; t < 2 && ok; ++t) {
              if (kc >= 1 && !mbar_wait(s_free(t), (kc - 1) & 1, wc, 14)) { ok = false; break; }
              tc_fence_after();
              const uint64_t qdesc = sdesc_sw128(sQ + qb * 2 * Q_BYTES + t * Q_BYTES, 16, 1024);
#pragma unroll
              for (int k = 0; k < HD / 16; ++k) umma_bf16_ss(tS(t), qdesc + k * 2, kdesc + k * 2, idesc_s, k > 0);
              umma_commit(s_full(t));
            }
            if (ok) umma_commit(k_empty(st));
          }
          if (ok) umma_commit(q_empty(qb));  // the item's Q buffer is free once its S products are done
        }
      } else {
        constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, HD, true);  // B = V tile, MN-major, N = 64
        const int t = warp - 2;
        int vc = 0;  // V tiles consumed, across items
        for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
          const int n_kv = decode(w).n_kv;
          for (int j = 0; j < n_kv; ++j, ++vc) {
            const int st = vc % NV;
            if (!mbar_wait(v_full(st), (vc / NV) & 1, wc, 15) || !mbar_wait(p_full(t), vc & 1, wc, 16)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vdesc = sdesc_sw128(sV + st * KV_BYTES, 1024, 1024);
#pragma unroll
            for (int k = 0; k < BKV / 16; ++k)
              umma_bf16_ts(tO(t), tP(t) + 8 * k, vdesc + k * 128, idesc_o, (j > 0 || k > 0) ? 1u : 0u);
            umma_commit(pv_done(t));
            umma_commit(v_empty(st));
          }
        }
      }
      // Every MMA this thread issued completes before TMEM is released.
      umma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kSoftmaxRegs) : "memory");
    // ---------------- softmax / correction / output: one query row per thread
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    // The turn passes through two hardware named barriers of 256 threads: barrier 1 is tile A's
    // turn, barrier 2 tile B's. The four warps taking the turn sync, the four passing it arrive.
    // Per key tile, tile B syncs on 2 and arrives on 1; tile A syncs on 1 (from its second tile)
    // and arrives on 2; tile A closes with one more sync on 1. Both tiles walk the same key tiles,
    // so every phase completes. After a failed wait a warp runs the turn operations of the key
    // tiles it has not walked yet before it stops, so the other tile never waits for it in vain.
    bool ok = true;
    int g = 0;       // key tiles processed, across items
    int g_turn = 0;  // the first key tile whose turn operations have not run
    for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
      const int kv0 = decode(w).kv0, n_kv = decode(w).n_kv;
      float m = -CUDART_INF_F;  // running maximum, in units of scale_log2
      float l = 0.0f;           // running denominator
      for (int j = 0; j < n_kv; ++j, ++g) {
        if (!mbar_wait_warp(s_full(t), g & 1, wc, 17)) { ok = false; break; }
        tc_fence_after();
        float sv[128];
        {
          // the row's 128 scores: four loads in flight, one wait
          uint32_t r[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tS(t) + lane_off + c * 32, r[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) sv[c * 32 + e] = __uint_as_float(r[c][e]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free(t));  // the MMA may overwrite S with the next tile

        const int valid = T - (kv0 + j) * BKV;  // keys of this tile inside the window
        if (valid < BKV) {              // only a window's last tile can be partial (warp-uniform)
#pragma unroll
          for (int c = 0; c < 128; ++c) sv[c] = (c < valid) ? sv[c] : -CUDART_INF_F;
        }
        // Row maximum: eight independent chains of three-input max.
        float mc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float a = fmax3(sv[16 * k], sv[16 * k + 1], sv[16 * k + 2]);
#pragma unroll
          for (int e = 3; e < 15; e += 2) a = fmax3(a, sv[16 * k + e], sv[16 * k + e + 1]);
          mc[k] = fmaxf(a, sv[16 * k + 15]);
        }
        const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), fmax3(fmax3(mc[3], mc[4], mc[5]), mc[6], mc[7]));
        const float mx_s = mx * scale_log2;
        const float m_new = (mx_s > m + kRescaleThreshold) ? mx_s : m;
        const float alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)

        // Ping-pong: the two tiles take turns on the exponentials (MUFU), so that one tile's
        // exponentials overlap the other tile's loads, stores and waits instead of contending.
        // Tile A's turn j follows tile B's exponentials of tile j-1; tile B's follows A's of j.
        if (t == 1 || g > 0) named_sync(1 + t, 256);

        // p = 2^(s * scale_log2 - m_new): packed fp32x2 FMA for the argument, packed adds for the
        // row sum; P is packed to bf16 pairs before waiting on the previous PV product.
        const uint64_t c2 = pack_f32x2(scale_log2, scale_log2);
        const uint64_t nm2 = pack_f32x2(-m_new, -m_new);
        uint64_t sum2a = pack_f32x2(0.0f, 0.0f), sum2b = sum2a;
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
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
        __syncwarp();
        named_arrive(2 - t, 256);  // the other tile's turn
        g_turn = g + 1;

        if (j > 0) {
          // PV[j-1] must be complete: P is overwritten below and O may be rescaled.
          if (!mbar_wait_warp(pv_done(t), (g - 1) & 1, wc, 18)) { ok = false; break; }
          tc_fence_after();
          if (__any_sync(0xffffffffu, m_new != m)) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(tO(t) + lane_off + half * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tmem_st_32x32b_x32(tO(t) + lane_off + half * 32, o);
            }
            tmem_st_wait();
          }
        }

        // P row (128 keys as 64 bf16 pairs) into the tile's P columns of TMEM.
        {
          uint32_t p0[32], p1[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            p0[e] = pk[e];
            p1[e] = pk[32 + e];
          }
          tmem_st_32x32b_x32(tP(t) + lane_off, p0);
          tmem_st_32x32b_x32(tP(t) + lane_off + 32, p1);
          tmem_st_wait();
        }
        l = l * alpha + sum;
        m = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(t));
      }
      if (!ok) break;
      if (!mbar_wait_warp(pv_done(t), (g - 1) & 1, wc, 19)) { ok = false; break; }
      {
        // The item's output, from O in TMEM once the PV product of its last key tile is done;
        // the next item's first PV product (which overwrites O) waits for P that this warp
        // writes only after these reads.
        tc_fence_after();
        const Item it = decode(w);
        const int tq_row = it.q0 + t * BQ + row;
        if (n_splits == 1) {
          const float inv_l = 1.0f / l;
          uint16_t* dst = out + (static_cast<size_t>(it.b) * T + tq_row) * out_stride + it.h * HD;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO(t) + lane_off + half * 32, o);
            tmem_ld_wait();
            if (tq_row < T && in_bounds(it.b < n_windows && it.h * HD + HD <= out_stride, err, 73)) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + half * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float* f = reinterpret_cast<const float*>(o) + q * 8;
                d4[q] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l), pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                                   pack_bf16x2(f[4] * inv_l, f[5] * inv_l), pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
              }
            }
          }
        } else {
          // Split keys: keep this split's unnormalised numerator, its reference maximum m (log2
          // units, scores pre-scaled) and its denominator l for the combine kernel.
          const size_t pi = (static_cast<size_t>(it.b * H + it.h) * n_splits + it.split) * T + tq_row;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO(t) + lane_off + half * 32, o);
            tmem_ld_wait();
            if (tq_row < T && in_bounds(pi < static_cast<size_t>(n_splits) * n_windows * H * T, err, 74)) {
              float4* d4 = reinterpret_cast<float4*>(part_o + pi * HD + half * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                d4[q] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                    __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
            }
          }
          if (tq_row < T) part_ml[pi] = make_float2(m, l);
        }
      }
    }
    if (!ok) {
      int n_tiles = 0;
      for (int w = blockIdx.x; w < n_items; w += gridDim.x) n_tiles += decode(w).n_kv;
      for (int gg = g_turn; gg < n_tiles; ++gg) {
        if (t == 1 || gg > 0) named_sync(1 + t, 256);
        named_arrive(2 - t, 256);
      }
    }
    if (t == 0) named_sync(1, 256);  // tile B's last hand-over
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Merge of the key splits of one (window, head, query row): with per-split maximum m_s,
// denominator l_s and numerator O_s, m = max_s m_s and
//   o = sum_s 2^(m_s - m) O_s / sum_s 2^(m_s - m) l_s
// (the chunked merge of oxinfer 0.0.5 src/whisper/model.rs, CrossLayer::attend: per-chunk
// maximum, sum and partial product, combined with exp(m_c - m) weights). Sixteen lanes per
// (row, head), four output columns each.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part_o,
                                                           const float2* __restrict__ part_ml,
                                                           uint16_t* __restrict__ out, int out_stride, int B,
                                                           int T, int H, int n_splits) {
  pdl_trigger();
  pdl_wait();
  const long long pair = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int c4 = threadIdx.x & 15;
  if (pair >= static_cast<long long>(B) * H * T) return;
  const int t = static_cast<int>(pair % T);
  const int h = static_cast<int>((pair / T) % H);
  const int b = static_cast<int>(pair / (static_cast<long long>(T) * H));
  const size_t base = static_cast<size_t>(b * H + h) * n_splits;
  float mmax = -CUDART_INF_F;
  for (int sp = 0; sp < n_splits; ++sp) mmax = fmaxf(mmax, part_ml[(base + sp) * T + t].x);
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int sp = 0; sp < n_splits; ++sp) {
    const size_t pi = (base + sp) * T + t;
    const float2 ml = part_ml[pi];
    const float wgt = ex2_approx(ml.x - mmax);
    const float4 o = reinterpret_cast<const float4*>(part_o + pi * HD)[c4];
    num.x += wgt * o.x; num.y += wgt * o.y; num.z += wgt * o.z; num.w += wgt * o.w;
    den += wgt * ml.y;
  }
  const float inv = 1.0f / den;
  uint16_t* dst = out + (static_cast<size_t>(b) * T + t) * out_stride + h * HD + 4 * c4;
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(num.x * inv, num.y * inv), pack_bf16x2(num.z * inv, num.w * inv));
}

}  // namespace

namespace wenc_host {

int attention_pick_splits(int B, int T, int H, int num_sms) {
  const long long ctas = static_cast<long long>((T + 2 * kAttnBQ - 1) / (2 * kAttnBQ)) * H * B;
  const int n_kv = (T + kAttnBKV - 1) / kAttnBKV;
  if (2 * ctas > num_sms || n_kv < 2) return 1;
  int s = static_cast<int>(num_sms / ctas);
  if (s > n_kv) s = n_kv;
  // equal tile counts per split, none empty
  const int tps = (n_kv + s - 1) / s;
  return (n_kv + tps - 1) / tps;
}

size_t attention_partial_bytes(int B, int T, int H, int n_splits) {
  if (n_splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(n_splits) * B * H * T;
  return rows * kAttnHD * sizeof(float) + rows * sizeof(float2);
}

static int clamp_splits(int T, int n_splits) {
  const int n_kv = (T + BKV - 1) / BKV;
  if (n_splits < 1) n_splits = 1;
  if (n_splits > n_kv) n_splits = n_kv;
  const int tps = (n_kv + n_splits - 1) / n_splits;
  return (n_kv + tps - 1) / tps;  // no empty split
}

cudaError_t launch_attention_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int q_col0,
                                  int k_col0, int v_col0, uint16_t* out, int out_stride, int B, int T, int H,
                                  uint32_t* err, cudaStream_t stream, int n_splits, float* part_o, float2* part_ml,
                                  int stop_after) {
  if (B <= 0 || T <= 0 || H <= 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Shared-memory opt-in, once per device (a repeat by a racing host thread is harmless).
  static std::atomic<int> configured_device{-1};
  if (configured_device.load(std::memory_order_acquire) != dev) {
    e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
    if (e != cudaSuccess) return e;
    configured_device.store(dev, std::memory_order_release);
  }
  // The softmax warpgroups' register increase is met only from the registers the CTA was
  // launched with: refuse to launch a build that was given fewer (a property of the build).
  static const int launch_regs = [] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, attn_fwd_kernel) == cudaSuccess ? fa.numRegs : 0;
  }();
  if (launch_regs * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  int num_sms = 0;
  e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  if (!part_o || !part_ml) n_splits = 1;
  n_splits = clamp_splits(T, n_splits);
  const int n_kv = (T + BKV - 1) / BKV;
  const int tps = (n_kv + n_splits - 1) / n_splits;
  const long long items = static_cast<long long>((T + 2 * BQ - 1) / (2 * BQ)) * n_splits * H * B;
  if (items > (1LL << 30)) return cudaErrorInvalidValue;
  // Persistent: one CTA per SM (shared memory and TMEM allow no second), each walking the items
  // w = blockIdx.x + k * gridDim.x.
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  return launch_pdl(attn_fwd_kernel, dim3(grid), dim3(kThreads), SMEM, stream, tq, tk, tv, q_col0, k_col0, v_col0,
                    out, out_stride, T, H, static_cast<int>(items), scale_log2, n_splits, tps, part_o, part_ml, err,
                    stop_after);
}

cudaError_t launch_attention_combine(const float* part_o, const float2* part_ml, uint16_t* out, int out_stride, int B,
                                     int T, int H, int n_splits, cudaStream_t stream) {
  n_splits = clamp_splits(T, n_splits);
  if (n_splits == 1 || B <= 0 || T <= 0 || H <= 0) return cudaSuccess;
  const long long threads = static_cast<long long>(B) * H * T * 16;
  return launch_pdl(attn_combine_kernel, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0, stream,
                    part_o, part_ml, out, out_stride, B, T, H, n_splits);
}

int attention_launches(int T, int n_splits) { return clamp_splits(T, n_splits) > 1 ? 2 : 1; }

cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int q_col0,
                             int k_col0, int v_col0, uint16_t* out, int out_stride, int B, int T, int H,
                             uint32_t* err, cudaStream_t stream, int n_splits, float* part_o, float2* part_ml) {
  if (!part_o || !part_ml) n_splits = 1;
  cudaError_t e = launch_attention_main(tq, tk, tv, q_col0, k_col0, v_col0, out, out_stride, B, T, H, err, stream,
                                        n_splits, part_o, part_ml);
  if (e != cudaSuccess) return e;
  return launch_attention_combine(part_o, part_ml, out, out_stride, B, T, H, n_splits, stream);
}

}  // namespace wenc_host
