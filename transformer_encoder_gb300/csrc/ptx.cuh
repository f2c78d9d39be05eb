// ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers with bounded waits, TMA tensor loads, and the tcgen05 family (TMEM
// allocation, UMMA issue/commit, TMEM loads/stores, ordering fences).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace wenc_dev {

// Device error word codes (low byte = wenc_status, next byte = the wait or check site).
constexpr uint32_t kErrTimeout = 5u;
constexpr uint32_t kErrIndex = 4u;  // WENC_ERR_CUDA: an index check of the bounds-checked build failed

// Index checks of the bounds-checked build (compiled with -DWENC_BOUNDS_CHECK): a checked access
// runs only if in_bounds() returns true; when its condition fails, the kernel records
// kErrIndex | site << 8 in the device error word and skips the access (no trap, no early return,
// so every barrier, wait and TMEM release of the kernel still happens). In the normal build the
// checks compile to nothing.
#ifdef WENC_BOUNDS_CHECK
__device__ __forceinline__ bool in_bounds(bool ok, uint32_t* err, uint32_t site) {
  if (!ok) *reinterpret_cast<volatile uint32_t*>(err) = kErrIndex | (site << 8);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, uint32_t*, uint32_t) { return true; }
#endif
// A wait that has not completed after this long is treated as a stalled pipeline.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// One bounded probe of the phase with the given parity. The suspend-time hint lets the
// hardware park the thread (no instruction issue) until the phase completes or ~1 ms
// passes, so waiting warps do not steal issue slots from the ones doing work.
constexpr uint32_t kSuspendHintNs = 1000000u;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Non-suspending test of the phase with the given parity (cheap when it has completed).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state for bounded waits inside one CTA: `abort_flag` (shared memory) tells
// every role to stop once any wait of the CTA has run out; `err` is the device error word.
struct WaitCtx {
  volatile uint32_t* abort_flag;
  uint32_t* err;
};

// Wait for the phase with the given parity to complete. Returns false (and raises the
// CTA's abort flag and the device error word) after kWaitLimitNs, or as soon as another
// role of the CTA has aborted; never spins forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
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

// Warp-collective form: every lane waits, then the warp agrees on the outcome, so the
// lanes stay converged for the .sync.aligned tcgen05 instructions that follow.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  const bool ok = mbar_wait(bar, parity, w, site);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (used only to drain in-flight copies on the
// error path before the CTA exits).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy (UMMA reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05: TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05: UMMA
// Shared-memory matrix descriptor for a tile stored with the 128-byte swizzle: rows of
// 128 bytes, 8-row atoms of 1024 bytes. `lbo`/`sbo` in bytes. Fields: start address>>4
// [0,14), leading byte offset>>4 [16,30), stride byte offset>>4 [32,46), descriptor
// version 1 [46,48), swizzle mode 2 = 128B [61,64).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A and B and an fp32 accumulator.
// D format [4,6) = 1 (f32); A format [7,10) = 1 (bf16); B format [10,13) = 1 (bf16);
// A major [15] = 0 (K-major); B major [16]; N>>3 [17,23); M>>4 [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Round an fp32 value to TF32 (10 explicit mantissa bits), to nearest with ties away from zero;
// the result is an fp32 value whose low 13 mantissa bits are zero, read exactly by kind::tf32.
__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Instruction descriptor, kind::tf32 with fp32 A and B in shared memory (read as TF32) and an
// fp32 accumulator: A and B format [7,10) / [10,13) = 2 (TF32), both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int m, int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every UMMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// ------------------------------------------------------------------ tcgen05: TMEM <-> registers
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base+i),
// columns col .. col+31. The warp may only touch its lane quadrant (warp_id % 4).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start while the previous kernel
// of the stream is still running. It must call pdl_wait() before its first global-memory access
// (the wait returns once the previous grid has completed and its writes are visible), and calls
// pdl_trigger() once every resource it allocates at start-up is held, so that the next kernel's
// CTAs can be scheduled and run their own set-up meanwhile.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ row statistics
// Mean and M2 (sum of squared deviations) of 32 values held four per lane by the 8 lanes of an
// aligned lane group (lane & 7 = position of the lane's four values). Two passes; every
// operation explicitly rounded, so two kernels that call this on the same values get the same
// bits (the GEMM epilogue that writes the residual stream and the row-statistics kernel).
__device__ __forceinline__ void chunk_stats32(float4 v, float& mean, float& m2) {
  float sm = __fadd_rn(__fadd_rn(v.x, v.y), __fadd_rn(v.z, v.w));
  sm = __fadd_rn(sm, __shfl_xor_sync(0xffffffffu, sm, 1));
  sm = __fadd_rn(sm, __shfl_xor_sync(0xffffffffu, sm, 2));
  sm = __fadd_rn(sm, __shfl_xor_sync(0xffffffffu, sm, 4));
  mean = __fmul_rn(sm, 1.0f / 32.0f);
  const float dx = __fsub_rn(v.x, mean), dy = __fsub_rn(v.y, mean), dz = __fsub_rn(v.z, mean),
              dw = __fsub_rn(v.w, mean);
  float q = __fadd_rn(__fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy)), __fadd_rn(__fmul_rn(dz, dz), __fmul_rn(dw, dw)));
  q = __fadd_rn(q, __shfl_xor_sync(0xffffffffu, q, 1));
  q = __fadd_rn(q, __shfl_xor_sync(0xffffffffu, q, 2));
  q = __fadd_rn(q, __shfl_xor_sync(0xffffffffu, q, 4));
  m2 = q;
}

// Merge the statistics (cm, cq) of chunk c (32 values) into those of chunks 0 .. c-1 (the
// pairwise update of Chan, Golub and LeVeque for combining sample means and M2).
__device__ __forceinline__ void chunk_merge32(float& mean, float& m2, float cm, float cq, int c) {
  if (c == 0) {
    mean = cm;
    m2 = cq;
    return;
  }
  const float na = 32.0f * c, nt = __fadd_rn(na, 32.0f);
  const float delta = __fsub_rn(cm, mean);
  mean = __fadd_rn(mean, __fmul_rn(delta, __fdiv_rn(32.0f, nt)));
  m2 = __fadd_rn(__fadd_rn(m2, cq), __fmul_rn(__fmul_rn(delta, delta), __fdiv_rn(__fmul_rn(na, 32.0f), nt)));
}

// ------------------------------------------------------------------ math helpers
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed fp32 pairs (one 64-bit register pair; .x in the low half).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace wenc_dev
