// gemm.cu -- the block's four contractions on the 5th-generation tensor cores.
//
// C[M, N] = A[M, K] . W[N, K]^T with the epilogue fused (the matmul_bias step of
// turbospark-runtime src/whisper/metal.rs encode_layer, with its separate add and
// gelu_erf passes folded in; inferencelayer src/whisper_gpu.rs WhisperEncoderGpu::forward
// fuses bias + GELU into its fc1 GEMM the same way):
//   QKV:      bf16 out = A W^T + b             (b's K slot is zero)
//   fc1:      bf16 out = GELU_erf(A W^T + b)
//   out, fc2: f32  out = resid + (A W^T + b)   (the residual add, in place on x)
//   conv2:    f32  out = GELU_erf(A W^T + b) + table[row % period]   (the stem's last
//             convolution with its positional rows, turbospark-runtime encode_partial)
//   cross K/V: bf16 out = A W^T + b written as planes: columns [p*P, (p+1)*P) of the product go
//             to plane p, a row-major [M, P] matrix (turbospark-runtime build_cross_caches: one K
//             and one V matrix per decoder layer)
// The TF32 form of the kernel takes fp32 A and W (already rounded to TF32 by their producers)
// and runs kind::tf32 MMAs (128 x BN x 8); its QKV and fc1 outputs are fp32 rounded to TF32.
//
// Design (sm_103a): persistent CTAs, one per SM, walk 128 x BN output tiles. Warp 0 is the
// TMA producer (A and W tiles, 128-byte swizzle, a STAGES-deep mbarrier ring); warp 1
// allocates TMEM and one of its threads issues tcgen05.mma (128 x BN x 16, bf16 in, fp32
// accumulate) into one of two TMEM accumulators; warps 2-9 drain the other accumulator
// (tcgen05.ld -> bias / GELU / residual -> global) while the next tile is being computed.
// The bf16 256-column GEMMs run the same roles on CTA pairs (clusters of two): a pair walks
// 256 x 256 tiles, its even CTA issuing M256 MMAs (cta_group::2) over both CTAs' shared memory,
// each CTA holding half of the W tile, so that five 32 KB stages fit with room to spare.
#include <cuda_bf16.h>
#include <stdlib.h>

#include <atomic>

#include "launch.h"
#include "ptx.cuh"

namespace {

using namespace wenc_dev;

constexpr int BM = wenc_host::kGemmBM;
constexpr int BK = wenc_host::kGemmBK;
constexpr int kEpiWarps = 8;                // two warps per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer warp, MMA warp, epilogue warps

// PAIR: a CTA pair (a cluster of two on one TPC) computes a 256 x BN tile with M256 MMAs
// (tcgen05 cta_group::2): each CTA holds its 128 rows of A and BN / 2 rows of W per stage, the
// pair's even CTA issues the MMAs, and each CTA's TMEM receives its own 128 rows. Half of W per
// CTA makes a stage 32 KB. Five stages: six fit, but five measured faster in the 32-block step
// (+0.5 to +0.9% in four A/B pairs on one box; four stages slowed fc2 by 10%).
template <int BN, bool PAIR = false>
struct GemmCfg {
  static constexpr int STAGES = PAIR ? 5 : (BN == 256) ? 4 : 6;
  // One stage holds 128-byte rows: 64 bf16 or 32 fp32 elements of K.
  static constexpr uint32_t A_BYTES = BM * 128;
  static constexpr uint32_t B_BYTES = (PAIR ? BN / 2 : BN) * 128;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two fp32 accumulators of BN columns
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 6;
  static constexpr uint32_t EPI_STAGE_BYTES = 32 * 32 * 4;  // one warp's 32 x 32 fp32 chunk
  static constexpr uint32_t EPI_BYTES = kEpiWarps * EPI_STAGE_BYTES;
  static constexpr size_t SMEM = 1024 /*align slack*/ + STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16;
};

// GELU(z) = z * Phi(z) = 0.5 z (1 + erf(z / sqrt(2))), with erf from the rational
// approximation of Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26:
//   erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),  t = 1 / (1 + p x),  x >= 0,
// |error| <= 1.5e-7, far below the bf16 rounding (2^-9 relative) of the fc1 output it feeds.
// erf is odd, so erf(-x) = -erf(x). Two MUFU operations (reciprocal, exp2) per value; evaluated
// on two values at once, the polynomial and the products as packed fp32x2 operations (one
// instruction per pair).
__device__ __forceinline__ void gelu_erf_x2(float& z0, float& z1) {
  const float x0 = fabsf(z0) * 0.70710678118654752f, x1 = fabsf(z1) * 0.70710678118654752f;
  float t0, t1;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t0) : "f"(fmaf(0.3275911f, x0, 1.0f)));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t1) : "f"(fmaf(0.3275911f, x1, 1.0f)));
  const uint64_t t = pack_f32x2(t0, t1);
  uint64_t poly = fma_f32x2(t, pack_f32x2(1.061405429f, 1.061405429f), pack_f32x2(-1.453152027f, -1.453152027f));
  poly = fma_f32x2(t, poly, pack_f32x2(1.421413741f, 1.421413741f));
  poly = fma_f32x2(t, poly, pack_f32x2(-0.284496736f, -0.284496736f));
  poly = fma_f32x2(t, poly, pack_f32x2(0.254829592f, 0.254829592f));
  poly = mul_f32x2(poly, t);
  const uint64_t xx = pack_f32x2(x0, x1);
  float a0, a1;
  unpack_f32x2(mul_f32x2(mul_f32x2(xx, xx), pack_f32x2(-1.4426950408889634f, -1.4426950408889634f)), a0, a1);
  const uint64_t neg_e = pack_f32x2(-ex2_approx(a0), -ex2_approx(a1));  // -exp(-x^2)
  float r0, r1;
  unpack_f32x2(fma_f32x2(poly, neg_e, pack_f32x2(1.0f, 1.0f)), r0, r1);  // erf(|x|)
  const uint64_t one_p = pack_f32x2(1.0f + copysignf(r0, z0), 1.0f + copysignf(r1, z1));  // 1 + erf(x)
  unpack_f32x2(mul_f32x2(mul_f32x2(pack_f32x2(z0, z1), pack_f32x2(0.5f, 0.5f)), one_p), z0, z1);
}

// ---- CTA-pair forms (cluster of two CTAs; every tcgen05 instruction of a pair kernel uses
// cta_group::2, as the PTX ISA requires one cta_group value per kernel)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of both CTAs; release / acquire at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrivals with relaxed semantics: they order nothing but the arrival itself (see release_acc).
__device__ __forceinline__ void mbar_arrive_relaxed_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Count `bytes` as arrived on this CTA's barrier without a copy (for a copy that was expected but
// never issued).
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Bounded wait (as mbar_wait) that acquires at cluster scope: for barriers the peer CTA arrives on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((n & 3u) == 0) {
      if (*w.abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *w.abort_flag = 1u;
        *reinterpret_cast<volatile uint32_t*>(w.err) = kErrTimeout | (site << 8);
        return false;
      }
    }
  }
}
// TMA tile load into this CTA's shared memory whose completion is counted on `bar_cluster`,
// a barrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (both CTAs' TMEM at d_tmem) (+)= A (each CTA's 128 rows) * B^T (BN / 2 rows from each CTA).
__device__ __forceinline__ void umma_bf16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at offset `bar` of every CTA in `cta_mask` when the MMAs issued so
// far have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(cta_mask)
               : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// The epilogue moves each warp's 32-row x 32-column accumulator chunk through a 4 KB
// shared-memory tile: thread r of the warp writes row r (as read from TMEM), then lane l
// reads rows 4i + l/8, columns 4(l%8)..4(l%8)+3, so every global load and store of the warp
// covers whole 128-byte row segments. 16-byte granules are XOR-swizzled by (row % 8), which
// keeps both the row-wise writes and the segment-wise reads free of bank conflicts.
__device__ __forceinline__ uint32_t stage_addr(uint32_t stage, int row, int granule) {
  return stage + row * 128 + ((granule ^ (row & 7)) << 4);
}

// Residual (or table) values this lane will need for one chunk (rows grow0 + 4i + lane/8).
// With period > 0 output row r reads table row r % period.
__device__ __forceinline__ void load_resid(float4 (&rr)[8], const float* resid, int grow0, int M, int N, int col,
                                           int lane, int period) {
  const int sub = lane >> 3, cl = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int grow = grow0 + 4 * i + sub;
    const int srow = period > 0 ? grow % period : grow;
    if (grow < M) rr[i] = *reinterpret_cast<const float4*>(resid + static_cast<size_t>(srow) * N + col + 4 * cl);
  }
}

// Per-row state of the LayerNorm-related epilogues for the eight rows (4i + lane/8) a lane
// handles in every chunk of a tile: the folded LayerNorm's mean and 1/std (EPI 5), or the
// running (mean, M2) of the row segment being written (EPI 7).
struct RowState {
  float a[8], b[8];
};

// EPI 0 = bias, 1 = bias + GELU, 2 = residual + bias (fp32 out), 3 = GELU(bias) + table row
// (fp32 out), 4 = bias with planar output (plane width `plane`), 5 = LayerNorm folded in
// (rstd (acc - mean colsum) + bias, bf16 out), 7 = as 2, plus a bf16 copy and the row
// segment's statistics. For EPI 0, 1 and 4 the output is bf16 (F32OUT false) or fp32 rounded
// to TF32 (F32OUT true: the operand of a TF32 GEMM). `chunk` is the chunk's index within the
// warp's column segment (EPI 7 merges the chunk statistics in that order).
template <int EPI, bool F32OUT>
__device__ __forceinline__ void epilogue_chunk(const uint32_t (&acc)[32], uint32_t stage, int lane, int grow0, int M,
                                               int N, int col, const float* __restrict__ bias,
                                               const float4 (&rr)[8], void* out, int plane,
                                               const wenc_host::GemmExtra& ex, RowState& rs, int chunk,
                                               uint32_t* err) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    st_shared_v4(stage_addr(stage, lane, q), acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  __syncwarp();
  const int sub = lane >> 3, cl = lane & 7;
  const float4 bb = __ldg(reinterpret_cast<const float4*>(bias + col) + cl);
  float4 cs = make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (EPI == 5) cs = __ldg(reinterpret_cast<const float4*>(ex.colsum + col) + cl);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + sub;
    const float4 a = ld_shared_f4(stage_addr(stage, r, cl));
    const int grow = grow0 + r;
    float4 v = make_float4(a.x + bb.x, a.y + bb.y, a.z + bb.z, a.w + bb.w);
    if constexpr (EPI == 5) {
      const float mu = rs.a[i], rstd = rs.b[i];
      v = make_float4(fmaf(rstd, fmaf(-mu, cs.x, a.x), bb.x), fmaf(rstd, fmaf(-mu, cs.y, a.y), bb.y),
                      fmaf(rstd, fmaf(-mu, cs.z, a.z), bb.z), fmaf(rstd, fmaf(-mu, cs.w, a.w), bb.w));
    }
    if constexpr (EPI == 7) {
      v = make_float4(rr[i].x + v.x, rr[i].y + v.y, rr[i].z + v.z, rr[i].w + v.w);
      // statistics of this row's 32 columns (8 lanes x 4 values), merged into the segment's
      // running (mean, M2) in chunk order
      float cm, cq;
      chunk_stats32(v, cm, cq);
      chunk_merge32(rs.a[i], rs.b[i], cm, cq, chunk);
    }
    if (grow < M && in_bounds(grow >= 0 && col >= 0 && col + 4 * cl + 4 <= N, err, 66)) {
      size_t off = static_cast<size_t>(grow) * N + col + 4 * cl;
      if constexpr (EPI == 4) {  // the chunk's 32 columns lie in one plane (plane % 32 == 0)
        const int pl = col / plane;
        off = (static_cast<size_t>(pl) * M + grow) * plane + (col - pl * plane) + 4 * cl;
      }
      if constexpr (EPI == 2 || EPI == 7) {
        if constexpr (EPI == 2) v = make_float4(rr[i].x + v.x, rr[i].y + v.y, rr[i].z + v.z, rr[i].w + v.w);
        *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = v;
        if constexpr (EPI == 7)
          *reinterpret_cast<uint2*>(ex.copy + off) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      } else if constexpr (EPI == 3) {
        gelu_erf_x2(v.x, v.y);
        gelu_erf_x2(v.z, v.w);
        v = make_float4(v.x + rr[i].x, v.y + rr[i].y, v.z + rr[i].z, v.w + rr[i].w);
        *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = v;
      } else {
        if constexpr (EPI == 1) {
          gelu_erf_x2(v.x, v.y);
          gelu_erf_x2(v.z, v.w);
        }
        if constexpr (F32OUT)
          *reinterpret_cast<float4*>(static_cast<float*>(out) + off) =
              make_float4(round_tf32(v.x), round_tf32(v.y), round_tf32(v.z), round_tf32(v.w));
        else
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + off) =
              make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      }
    }
  }
  __syncwarp();  // the stage is rewritten by the next chunk
}

// How one launch divides its output tiles among its scheduling units (CTAs, or CTA pairs), the
// same sequence for every role of a unit: whole tiles unit + i G (G = the number of units) over
// the first n_dp tiles; then, when the launch splits its last partial wave (tail_halves), one
// half-width unit each: the n_tail = num_tiles % G remaining tiles become 2 n_tail units of
// BN / 2 columns (an M128 (pair: M256) N(BN/2) product over the whole K), unit u < 2 n_tail
// taking half u % 2 of tile n_dp + u / 2. Each output element is the same fixed-order dot product
// either way. The kernel and the host-side self-test run this same code.
struct TileSchedule {
  int unit, n_units, n_dp, n_mine;
  bool has_unit;
  __host__ __device__ TileSchedule(int num_tiles, int unit_, int n_units_, bool tail_halves)
      : unit(unit_), n_units(n_units_) {
    const int n_tail = tail_halves ? num_tiles % n_units : 0;
    n_dp = num_tiles - n_tail;
    n_mine = (unit < n_dp) ? (n_dp - 1 - unit) / n_units + 1 : 0;
    has_unit = unit < 2 * n_tail;
  }
  // item i of this unit: its tile and, for the half-width unit, which half (-1: the whole tile)
  __host__ __device__ bool item(int i, int& tile, int& half) const {
    if (i < n_mine) {
      tile = unit + i * n_units;
      half = -1;
      return true;
    }
    if (i == n_mine && has_unit) {
      tile = n_dp + unit / 2;
      half = unit % 2;
      return true;
    }
    return false;
  }
};

// The size of a launch: one unit per tile, at most max_units; a last partial wave that would
// leave at least half of the units idle runs as twice as many half-width units (all tiles, when
// there are at most half as many tiles as units).
struct LaunchPlan {
  int units;
  int halves;
};
inline LaunchPlan plan_launch(int tiles, int max_units) {
  LaunchPlan p;
  p.units = tiles < max_units ? tiles : max_units;
  const int n_tail = tiles < max_units ? tiles : tiles % max_units;
  p.halves = (n_tail > 0 && 2 * n_tail <= max_units) ? 1 : 0;
  if (p.halves && tiles < max_units) p.units = 2 * tiles;
  return p;
}

template <int BN, int EPI, bool TF32, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmWh, int half_box, int M, int N,
                   int K, const float* __restrict__ bias, const float* resid, void* out, uint32_t* err,
                   int row_period, const wenc_host::GemmExtra ex, int tail_halves) {
  static_assert(!PAIR || (!TF32 && BN == 256), "CTA pairs run the bf16 256-column tiles");
  using C = GemmCfg<BN, PAIR>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * C::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + C::EPI_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  // CTA pair: the odd CTA's producer reports how many stages it loaded (into peer_loads of the
  // even CTA, then one arrival on loads_bar), so that the even CTA can drain every copy of the
  // pair that may still be in flight before the pair's final barrier.
  const uint32_t loads_bar = bar0 + 8u * (2 * STAGES + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* peer_loads = tmem_slot + 2;
  const WaitCtx wc{abort_flag, err};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The scheduling unit: a CTA, or a CTA pair (rank 0 or 1 within it) working on 256-row tiles.
  constexpr int TM = PAIR ? 2 * BM : BM;  // output rows per tile
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int n_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int m_tiles = (M + TM - 1) / TM;
  const int n_tiles = N / BN;
  const int num_tiles = m_tiles * n_tiles;
  // Tile order. The block GEMMs walk n fastest: a wave of CTAs shares one A row block, and W
  // (at most 13 MB) stays in L2. The cross K/V product's W spans every decoder layer (210 MB at
  // large-v3 dims) and its 3.9 GB output streams through L2, so it walks groups of kGroupM row
  // blocks: within a group m is fastest, and the group sweeps every column block before the
  // next group starts. A wave then shares a few W tiles, the group's slice of A (64 x 128 rows)
  // stays in L2, and W is read m_tiles / kGroupM times instead of once per row block.
  constexpr bool kGrouped = (EPI == 4);
  constexpr int kGroupM = 64;
  auto tile_m = [&](int t) {
    if constexpr (!kGrouped) return t / n_tiles;
    const int g = t / (kGroupM * n_tiles), first = g * kGroupM;
    const int gs = min(kGroupM, m_tiles - first);
    return first + (t - g * kGroupM * n_tiles) % gs;
  };
  auto tile_n = [&](int t) {
    if constexpr (!kGrouped) return t % n_tiles;
    const int g = t / (kGroupM * n_tiles), first = g * kGroupM;
    const int gs = min(kGroupM, m_tiles - first);
    return (t - g * kGroupM * n_tiles) / gs;
  };
  constexpr int BKE = TF32 ? 32 : BK;  // K elements per stage (128-byte rows)
  const int k_blocks = K / BKE;
  // Work items of this unit (see TileSchedule)
  const TileSchedule sched(num_tiles, unit, n_units, tail_halves != 0);
  auto item = [&](int i, int& tile, int& half) -> bool { return sched.item(i, tile, half); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), PAIR ? 2 * kEpiWarps : kEpiWarps);  // one arrival per epilogue warp (of the pair)
    }
    mbar_init(drain_bar, 1);
    mbar_init(loads_bar, 1);
    *abort_flag = 0u;
    *peer_loads = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    if (half_box) tma_prefetch_desc(&tmWh);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) {
    __syncwarp();
    cluster_sync_all();  // both CTAs' barriers are initialised before either signals the other's
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();  // TMEM is held: the next kernel may be scheduled
  pdl_wait();     // the previous kernel's outputs (A, residual) are complete from here on

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;
    uint32_t loads = 0;  // stages this CTA has loaded
    bool ok = true;
    int tile, half;
    for (int i = 0; ok && item(i, tile, half); ++i) {
      // First A row and first W row of this CTA's loads. Single CTA: a whole tile loads BN rows of
      // W; a half-width unit BN / 2 rows through the half-box map (without one, BN rows from its
      // half's first column, rows past N reading as zeros, of which it multiplies the first
      // BN / 2). CTA pair: each CTA loads its own 128 rows of A and its share of W through the
      // half-box map (BN / 2 rows; BN / 4 of them in a half-width unit, the rest of the box
      // unused), counted on the even CTA's full barrier, which expects both CTAs' bytes.
      const int m0 = tile_m(tile) * TM + static_cast<int>(rank) * BM;
      const int n0 = tile_n(tile) * BN + (half > 0 ? BN / 2 : 0) +
                     (PAIR ? static_cast<int>(rank) * (half < 0 ? BN / 2 : BN / 4) : 0);
      const bool hb = half >= 0 && half_box;
      const uint32_t stage_bytes = hb ? C::A_BYTES + C::B_BYTES / 2 : C::STAGE_BYTES;
      if (!in_bounds(tile >= 0 && tile < num_tiles && n0 >= 0 && n0 < N && m0 >= 0, err, 64)) {
        *abort_flag = 1u;  // the tile schedule left the output: stop as a failed wait would
        ok = false;
        break;
      }
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (PAIR && rank != 0 && ex.stop_odd_after >= 0 && loads >= static_cast<uint32_t>(ex.stop_odd_after)) {
          // self-test: this producer gives up here as if a wait had run out (site 31)
          *abort_flag = 1u;
          *reinterpret_cast<volatile uint32_t*>(err) = kErrTimeout | (31u << 8);
          ok = false;
          break;
        }
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc, 1)) { ok = false; break; }
        if constexpr (PAIR) {
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
          const uint32_t lead_full = map_to_rank(full_bar(stage), 0);
          tma_load_2d_pair(sA + stage * C::A_BYTES, &tmA, lead_full, kb * BKE, m0);
          tma_load_2d_pair(sB + stage * C::B_BYTES, &tmWh, lead_full, kb * BKE, n0);
        } else {
          mbar_arrive_expect_tx(full_bar(stage), stage_bytes);
          tma_load_2d(sA + stage * C::A_BYTES, &tmA, full_bar(stage), kb * BKE, m0);
          tma_load_2d(sB + stage * C::B_BYTES, hb ? &tmWh : &tmW, full_bar(stage), kb * BKE, n0);
        }
        issued_mask |= 1u << stage;
        ++loads;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if constexpr (PAIR) {
      // Ordered drain of the pair's copies, on every exit: both CTAs' copies of a stage complete on
      // the even CTA's full barrier, and a producer reuses a stage only after the MMAs consumed it,
      // so the copies that may still be in flight are those of the last STAGES stages either CTA
      // loaded. The odd CTA reports its count; the even CTA waits for each of those stages, first
      // arming the ones only the odd CTA loaded (for the odd CTA's bytes) and cancelling the bytes
      // the odd CTA never sent for the ones only it armed. Neither CTA leaves the final cluster
      // barrier before this ends, so no copy lands in shared memory that has been released.
      if (rank != 0) {
        st_cluster_u32(map_to_rank(smem_u32(const_cast<uint32_t*>(peer_loads)), 0), loads);
        mbar_arrive_cluster(map_to_rank(loads_bar, 0));  // release: the count is visible with the arrival
      } else {
        uint32_t odd = loads;
        const uint64_t t0 = global_timer_ns();
        bool have = false;
        while (!(have = mbar_try_wait_cluster(loads_bar, 0)) && global_timer_ns() - t0 <= kWaitLimitNs) {
        }
        if (have) odd = *peer_loads;
        const uint32_t n = loads > odd ? loads : odd;
        for (uint32_t i = n > static_cast<uint32_t>(STAGES) ? n - STAGES : 0; i < n; ++i) {
          const int s = static_cast<int>(i % STAGES);
          if (i >= loads) mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
          else if (i >= odd) mbar_complete_tx(full_bar(s), C::STAGE_BYTES);
          mbar_wait_drain(full_bar(s), (i / STAGES) & 1u);
        }
      }
    } else if (!ok) {
      // Error path: let the copies already issued land before the CTA exits.
      for (int s = 0; s < STAGES; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        mbar_wait_drain(full_bar(s), par);
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- UMMA issuer (a pair's even CTA issues for both)
    // Four MMAs per stage, each over 32 bytes of K (16 bf16 or 8 TF32 elements).
    constexpr uint32_t idesc_full = TF32 ? idesc_tf32_f32(BM, BN) : idesc_bf16_f32(TM, BN, false);
    constexpr uint32_t idesc_half = TF32 ? idesc_tf32_f32(BM, BN / 2) : idesc_bf16_f32(TM, BN / 2, false);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int tile, half;
    for (int local = 0; ok && item(local, tile, half); ++local) {
      const uint32_t idesc = half < 0 ? idesc_full : idesc_half;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const bool freed = PAIR ? mbar_wait_cluster(tempty_bar(acc), acc_phase ^ 1u, wc, 2)
                              : mbar_wait(tempty_bar(acc), acc_phase ^ 1u, wc, 2);
      if (!freed) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, wc, 3)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_base = sA + stage * C::A_BYTES;
        const uint32_t b_base = sB + stage * C::B_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = sdesc_sw128(a_base + k * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(b_base + k * 32, 16, 1024);
          if constexpr (TF32) umma_tf32_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          else if constexpr (PAIR) umma_bf16_ss_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          else umma_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
        }
        if constexpr (PAIR) umma_commit_pair(empty_bar(stage), 0x3);  // both CTAs' stage is free
        else umma_commit(empty_bar(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if constexpr (PAIR) umma_commit_pair(tfull_bar(acc), 0x3);
      else umma_commit(tfull_bar(acc));
    }
    // Every UMMA issued by this thread completes before TMEM is released.
    if constexpr (PAIR) umma_commit_pair(drain_bar, 0x1);
    else umma_commit(drain_bar);
    mbar_wait_drain(drain_bar, 0);
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> registers -> shared -> global
    // Eight warps: warp w reads TMEM lane quadrant w % 4 (rows 32q..32q+31 of the tile) and
    // one half of the tile's columns, 32 columns at a time (see epilogue_chunk). For the
    // residual epilogue each lane keeps two chunks of residual loads in flight, continuing into
    // the next tile (the first tile's before its accumulator is ready). The TMEM buffer is
    // released as soon as its last chunk has been read.
    constexpr int CH = BN / 64;  // 32-column chunks per warp
    const int quad = warp & 3;
    const int col_half = (warp - 2) >> 2;
    const uint32_t stage = smem_u32(smem + STAGES * C::STAGE_BYTES) + (warp - 2) * C::EPI_STAGE_BYTES;
    auto row0_of = [&](int t) { return tile_m(t) * TM + static_cast<int>(rank) * BM + quad * 32; };
    // The barrier that frees an accumulator lives in the issuing CTA (the pair's even one). The
    // arrival is relaxed: all it orders is this warp's TMEM reads (complete at tcgen05.wait::ld,
    // and fenced by tcgen05.fence::before_thread_sync) before the next MMA overwrites the
    // accumulator; a release would also wait for the warp's earlier global stores of the tile to
    // be performed, stalling the epilogue for nothing.
    auto release_acc = [&](int a) {
      if constexpr (PAIR) mbar_arrive_relaxed_cluster(map_to_rank(tempty_bar(a), 0));
      else mbar_arrive_relaxed(tempty_bar(a));
    };
    auto col_of = [&](int t) { return tile_n(t) * BN + col_half * (BN / 2); };
    float4 rb[2][8];
    constexpr bool kRowInput = (EPI == 2 || EPI == 3 || EPI == 7);  // residual rows or table rows
    // A half-width unit's BN / 2 columns sit in TMEM columns [0, BN / 2) and belong to the warps
    // of the first column half; the other warps only release the buffer.
    auto cols_of = [&](int t, int hf) { return hf < 0 ? col_of(t) : tile_n(t) * BN + hf * (BN / 2); };
    auto active = [&](int hf) { return hf < 0 || col_half == 0; };
    int tile, half;
    if constexpr (kRowInput) {
      if (item(0, tile, half) && active(half)) {
        load_resid(rb[0], resid, row0_of(tile), M, N, cols_of(tile, half), lane, row_period);
        if (CH > 1) load_resid(rb[1], resid, row0_of(tile), M, N, cols_of(tile, half) + 32, lane, row_period);
      }
    }
    for (int local = 0; item(local, tile, half); ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int grow0 = row0_of(tile);
      const int c0 = cols_of(tile, half);
      int next, next_half;
      const bool prefetch_next = item(local + 1, next, next_half) && active(next_half);
      RowState rs;  // (EPI 5: loaded before the accumulator wait, to hide the load latency)
      if constexpr (EPI == 5) {
        // The folded LayerNorm's mean and 1/std of this lane's eight rows, from the producer's
        // segment statistics (equal-width segments: mean of the means, M2 by the parallel rule).
        // The 8 lanes that share a row split its segments (lane cl takes segments cl + 8 s,
        // s < 4: up to 32), issue all their loads together, and combine by shuffles in a fixed
        // order.
        const int nseg = K / ex.seg_w;
        const int sub = lane >> 3, cl = lane & 7;
        float2 sg[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int grow = min(grow0 + 4 * i + sub, M - 1);
          const float2* st = ex.stats + static_cast<size_t>(grow) * nseg;
#pragma unroll
          for (int q = 0; q < 4; ++q) sg[i][q] = cl + 8 * q < nseg ? st[cl + 8 * q] : make_float2(0.0f, 0.0f);
        }
        const float inv_nseg = 1.0f / nseg;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float msum = (sg[i][0].x + sg[i][1].x) + (sg[i][2].x + sg[i][3].x);
          msum += __shfl_xor_sync(0xffffffffu, msum, 1);
          msum += __shfl_xor_sync(0xffffffffu, msum, 2);
          msum += __shfl_xor_sync(0xffffffffu, msum, 4);
          const float mu = msum * inv_nseg;
          float m2 = 0.0f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float dq = sg[i][q].x - mu;
            if (cl + 8 * q < nseg) m2 += sg[i][q].y + ex.seg_w * dq * dq;
          }
          m2 += __shfl_xor_sync(0xffffffffu, m2, 1);
          m2 += __shfl_xor_sync(0xffffffffu, m2, 2);
          m2 += __shfl_xor_sync(0xffffffffu, m2, 4);
          rs.a[i] = mu;
          rs.b[i] = 1.0f / sqrtf(m2 / K + ex.eps);
        }
      }
      if (!mbar_wait_warp(tfull_bar(acc), acc_phase, wc, 4)) break;
      tc_fence_after();
      if (!active(half)) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(acc);
        continue;
      }
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN +
                             (half < 0 ? col_half * (BN / 2) : 0);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
        if (c == CH - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_acc(acc);
        }
        epilogue_chunk<EPI, TF32>(r, stage, lane, grow0, M, N, c0 + c * 32, bias, rb[c & 1], out, row_period, ex, rs,
                                  c, err);
        if constexpr (kRowInput) {
          if (c + 2 < CH) {
            load_resid(rb[c & 1], resid, grow0, M, N, c0 + (c + 2) * 32, lane, row_period);
          } else if (prefetch_next) {
            load_resid(rb[c & 1], resid, row0_of(next), M, N, cols_of(next, next_half) + (c + 2 - CH) * 32, lane,
                       row_period);
          }
        }
      }
      if constexpr (EPI == 7) {
        // this warp's column segment (BN / 2 columns) of its eight rows is complete
        const int sub = lane >> 3, cl = lane & 7;
        if (cl == 0) {
          const int nseg = N / ex.seg_w, seg = c0 / ex.seg_w;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int grow = grow0 + 4 * i + sub;
            if (grow < M) ex.stats_out[static_cast<size_t>(grow) * nseg + seg] = make_float2(rs.a[i], rs.b[i]);
          }
        }
      }
    }
  }

  tc_fence_before();
  if constexpr (PAIR) {
    // neither CTA frees its TMEM or shared memory while the other may still reach into them
    __syncwarp();
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int EPI, bool TF32>
cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmW, const CUtensorMap* tmW_half, int M, int N,
                       int K, const float* bias, const float* resid, void* out, uint32_t* err, int num_sms,
                       cudaStream_t stream, int row_period, const wenc_host::GemmExtra& ex) {
  using C = GemmCfg<BN>;
  auto kern = gemm_tc_kernel<BN, EPI, TF32, false>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Shared-memory opt-in, once per device and instantiation (a repeat by a racing host thread
  // is harmless).
  static std::atomic<int> configured_device{-1};
  if (configured_device.load(std::memory_order_acquire) != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    configured_device.store(dev, std::memory_order_release);
  }
  const LaunchPlan plan = plan_launch(((M + BM - 1) / BM) * (N / BN), num_sms);
  return wenc_host::launch_pdl(kern, dim3(plan.units), dim3(kThreads), C::SMEM, stream, tmA, tmW,
                               tmW_half ? *tmW_half : tmW, tmW_half ? 1 : 0, M, N, K, bias, resid, out, err,
                               row_period, ex, plan.halves);
}

// The CTA-pair form: clusters of two CTAs, as many pairs as fit at once (at most one CTA per
// SM), each walking 256-row tiles. tmW_half is W with a box of 128 rows (one CTA's half of W).
template <int EPI>
cudaError_t launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmW_half, int M, int N, int K, const float* bias,
                        const float* resid, void* out, uint32_t* err, int num_sms, cudaStream_t stream,
                        int row_period, const wenc_host::GemmExtra& ex) {
  using C = GemmCfg<256, true>;
  auto kern = gemm_tc_kernel<256, EPI, false, true>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // Shared-memory opt-in and the number of co-resident pairs, once per device and
  // instantiation (a repeat by a racing host thread is harmless).
  static std::atomic<int> max_pairs[64];
  int pairs_fit = max_pairs[dev].load(std::memory_order_acquire);
  if (pairs_fit <= 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&pairs_fit, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (pairs_fit <= 0) return cudaErrorInvalidConfiguration;
    max_pairs[dev].store(pairs_fit, std::memory_order_release);
  }
  const int max_units = pairs_fit < num_sms / 2 ? pairs_fit : num_sms / 2;
  if (max_units <= 0) return cudaErrorInvalidConfiguration;
  const LaunchPlan plan = plan_launch(((M + 255) / 256) * (N / 256), max_units);
  cfg.gridDim = dim3(2 * plan.units);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmW_half, tmW_half, 1, M, N, K, bias, resid, out, err, row_period, ex,
                            plan.halves);
}

// CTA pairs serve the bf16 256-column GEMMs that come with a half-height W map; the
// environment variable WENC_GEMM_PAIR=0 keeps them on single CTAs (for comparisons).
bool use_pair(bool tf32, int bn, int epilogue, const CUtensorMap* tmW_half) {
  static const bool enabled = [] {
    const char* v = getenv("WENC_GEMM_PAIR");
    return !(v && v[0] == '0');
  }();
  return enabled && !tf32 && bn == 256 && tmW_half != nullptr && epilogue != 4;
}

}  // namespace

namespace wenc_host {

bool gemm_pair_enabled() { return use_pair(false, 256, 0, reinterpret_cast<const CUtensorMap*>(1)); }

int gemm_schedule_cover(int M, int N, bool pair, int max_units, int* cover, int cover_len, int* unit_halves,
                        int* units_out, int* halves_out) {
  const int bn = pair ? 256 : gemm_pick_bn(N);
  if (M < 1 || bn == 0 || N % bn != 0 || max_units < 1) return -1;
  const int rows = pair ? 2 * BM : BM;
  const long long tiles_ll = static_cast<long long>((M + rows - 1) / rows) * (N / bn);
  if (tiles_ll > cover_len / 2) return -1;
  const int tiles = static_cast<int>(tiles_ll);
  const LaunchPlan plan = plan_launch(tiles, max_units);
  for (int i = 0; i < 2 * tiles; ++i) cover[i] = 0;
  for (int u = 0; u < plan.units; ++u) {
    const TileSchedule sched(tiles, u, plan.units, plan.halves != 0);
    int n = 0, tile, half;
    for (int i = 0; sched.item(i, tile, half); ++i) {
      if (tile < 0 || tile >= tiles) return -2;
      if (half < 0) {
        ++cover[2 * tile];
        ++cover[2 * tile + 1];
        n += 2;
      } else {
        ++cover[2 * tile + half];
        n += 1;
      }
    }
    if (unit_halves) unit_halves[u] = n;
  }
  *units_out = plan.units;
  *halves_out = plan.halves;
  return 0;
}

int gemm_pick_bn(int N) {
  if (N % 256 == 0) return 256;
  if (N % 128 == 0) return 128;
  return 0;
}

cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmW, int M, int N, int K, int bn, int epilogue,
                        const float* bias, const float* resid, void* out, uint32_t* err, int num_sms,
                        cudaStream_t stream, bool tf32, int row_period, const GemmExtra& ex,
                        const CUtensorMap* tmW_half) {
  if (M <= 0) return cudaSuccess;
  if (epilogue == 5 &&
      (!ex.colsum || !ex.stats || ex.seg_w <= 0 || K % ex.seg_w != 0 || K / ex.seg_w > 32 || tf32))
    return cudaErrorInvalidValue;
  if (epilogue == 7 && (!ex.copy || !ex.stats_out || ex.seg_w != bn / 2 || tf32)) return cudaErrorInvalidValue;
  if (epilogue == 3 && row_period <= 0) return cudaErrorInvalidValue;
  if (epilogue == 4 && (row_period <= 0 || row_period % 32 != 0 || N % row_period != 0)) return cudaErrorInvalidValue;
  if (use_pair(tf32, bn, epilogue, tmW_half)) {
    switch (epilogue) {
      case 0: return launch_pair<0>(tmA, *tmW_half, M, N, K, bias, resid, out, err, num_sms, stream, row_period, ex);
      case 1: return launch_pair<1>(tmA, *tmW_half, M, N, K, bias, resid, out, err, num_sms, stream, row_period, ex);
      case 2: return launch_pair<2>(tmA, *tmW_half, M, N, K, bias, resid, out, err, num_sms, stream, row_period, ex);
      case 3: return launch_pair<3>(tmA, *tmW_half, M, N, K, bias, resid, out, err, num_sms, stream, row_period, ex);
      case 5: return launch_pair<5>(tmA, *tmW_half, M, N, K, bias, resid, out, err, num_sms, stream, row_period, ex);
      case 7: return launch_pair<7>(tmA, *tmW_half, M, N, K, bias, resid, out, err, num_sms, stream, row_period, ex);
      default: break;
    }
  }
#define WENC_GEMM_CASE(BNV, EPIV, TF) \
  if (bn == BNV && epilogue == EPIV && tf32 == TF)                                        \
    return launch_one<BNV, EPIV, TF>(tmA, tmW, tmW_half, M, N, K, bias, resid, out, err, num_sms, stream, row_period, ex);
  WENC_GEMM_CASE(256, 0, false)
  WENC_GEMM_CASE(256, 1, false)
  WENC_GEMM_CASE(256, 2, false)
  WENC_GEMM_CASE(128, 0, false)
  WENC_GEMM_CASE(128, 1, false)
  WENC_GEMM_CASE(128, 2, false)
  WENC_GEMM_CASE(256, 3, false)
  WENC_GEMM_CASE(128, 3, false)
  WENC_GEMM_CASE(256, 4, false)
  WENC_GEMM_CASE(128, 4, false)
  WENC_GEMM_CASE(256, 5, false)
  WENC_GEMM_CASE(128, 5, false)
  WENC_GEMM_CASE(256, 7, false)
  WENC_GEMM_CASE(128, 7, false)
  WENC_GEMM_CASE(256, 0, true)
  WENC_GEMM_CASE(256, 1, true)
  WENC_GEMM_CASE(256, 2, true)
  WENC_GEMM_CASE(128, 0, true)
  WENC_GEMM_CASE(128, 1, true)
  WENC_GEMM_CASE(128, 2, true)
  WENC_GEMM_CASE(256, 3, true)
  WENC_GEMM_CASE(128, 3, true)
  WENC_GEMM_CASE(256, 4, true)
  WENC_GEMM_CASE(128, 4, true)
#undef WENC_GEMM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace wenc_host
