// launch.h -- host-side launchers of the kernels (internal to libwenc.so).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>

namespace wenc_host {

// Launch with programmatic stream serialisation (the kernel overlaps its set-up with the tail of
// the previous kernel in the stream; see pdl_wait / pdl_trigger in ptx.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Tensor-map construction (cuTensorMapEncodeTiled through the runtime's driver entry
// point, so the library does not link libcuda directly).
// 2-D bf16 view: `outer` rows of `inner` elements, rows `row_stride_bytes` apart; the box is
// box_inner x box_outer elements, 128-byte swizzled (box_inner * 2 must be 128).
bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, std::string* why);
// 2-D fp32 view, box box_inner x box_outer (box_inner * 4 must be 128).
bool make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                      uint32_t box_inner, uint32_t box_outer, std::string* why);
// 3-D bf16 view [dim2][dim1][inner] with explicit strides (bytes) for dims 1 and 2.
bool make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t dim1, uint64_t dim2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box_inner, uint32_t box1,
                       std::string* why);
// The same over fp32 elements (box_inner * 4 must be 128).
bool make_tmap_3d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t dim1, uint64_t dim2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box_inner, uint32_t box1,
                      std::string* why);

// ---------------------------------------------------------------- LayerNorm
bool layernorm_supported(int d);
// out_fmt: 0 = fp32, 1 = bf16, 2 = fp32 rounded to TF32.
cudaError_t launch_layernorm(const float* x, const float* w, const float* b, void* y, int rows, int d, float eps,
                             int out_fmt, cudaStream_t stream);

// Row statistics for a LayerNorm-folded GEMM (see GemmExtra): xb = bf16(x), stats [rows][d / seg]
// = (mean, M2) of each seg-column segment (seg 128 or 64).
cudaError_t launch_row_stats(const float* x, uint16_t* xb, float2* stats, int rows, int d, int seg, cudaStream_t stream);
// Fold a LayerNorm (ln_w, ln_b) into the GEMM after it (see fold_ln_kernel in ln.cu).
cudaError_t launch_fold_ln(const void* w, bool w_bf16, const float* ln_w, const float* ln_b, const float* bias,
                           uint16_t* wp, float* colsum, float* bias_out, int n_out, int k, cudaStream_t stream);

// ---------------------------------------------------------------- GEMM (tcgen05)
// C[M, N] = A[M, K] * W[N, K]^T with a fused epilogue (wenc_epilogue values).
// Tile: 128 x bn (bn = 256 or 128), k-block 64. tmA: box 64 x 128 over A; tmW: box 64 x bn over W.
int gemm_pick_bn(int N);  // 0 if N is unsupported
bool gemm_pair_enabled();   // bf16 256-column GEMMs run as CTA pairs (not switched off by WENC_GEMM_PAIR=0)
// Host-side replay of how a launch of M x N (single CTAs: 128-row tiles of gemm_pick_bn(N)
// columns; pair: 256 x 256 tiles) with at most max_units units divides its tiles, through the
// same schedule code the kernel runs. cover[2t + h] (cover_len >= 2 x tiles) counts how often
// column half h of tile t is computed; unit_halves[u] (max_units entries, or NULL) the half-tiles
// unit u computes. Returns 0, or < 0 for an unsupported shape or a short cover array.
int gemm_schedule_cover(int M, int N, bool pair, int max_units, int* cover, int cover_len, int* unit_halves,
                        int* units_out, int* halves_out);
constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;
// tf32 = false: bf16 A and W (maps with box 64 x rows), epilogues 0, 1, 2.
// tf32 = true: fp32 A and W read as TF32 (maps with box 32 x rows); epilogues 0 and 1 write
// fp32 rounded to TF32 instead of bf16. K must be a multiple of 64 (bf16) or 32 (TF32).
// Epilogue 3 (internal, the stem's conv2): out fp32 = GELU_erf(A W^T + bias) + resid[row % row_period]
// with resid a [row_period, N] fp32 table (row_period > 0).
constexpr int kEpiGeluTable = 3;
// LayerNorm folded into the GEMMs around it (the BF16 forward folds LN1 into QKV):
// - epilogue 5: out bf16 = rstd_r (acc - mu_r colsum_n) + bias_n, where the GEMM
//   ran on the raw residual stream x (bf16 copy) against W' = W diag(ln_w), colsum = row sums of W'
//   and bias = W ln_b + b, and (mu_r, rstd_r) come from the per-row segment statistics `stats`
//   ([M][K / seg_w] float2 = (segment mean, segment M2), each segment seg_w columns wide);
// - epilogue 7: as epilogue 2 (out fp32 = resid + acc + bias), and also writes `copy`, the output
//   rounded to bf16, and `stats_out`, the (mean, M2) of every seg_w-column row segment (seg_w =
//   bn / 2), which the next LN-folded GEMM reads.
struct GemmExtra {
  const float* colsum = nullptr;
  const float2* stats = nullptr;
  float2* stats_out = nullptr;
  uint16_t* copy = nullptr;
  float eps = 0.0f;
  int seg_w = 0;
  // Self-test only (wenc_selftest_gemm_pair_abort): in the CTA-pair form, the odd CTA's TMA
  // producer stops after this many stages and reports a timeout, as if one of its waits had run
  // out; -1 (every other caller) leaves the kernel unchanged.
  int stop_odd_after = -1;
};
constexpr int kEpiLnBias = 5;
constexpr int kEpiResidStats = 7;

// Epilogue 4 (internal, the cross K/V precompute): as epilogue 0, written as planes of width
// row_period: out[(col / P) * M * P + row * P + col % P]. P % 32 == 0 and N % P == 0.
constexpr int kEpiBiasPlanes = 4;
// tmW_half (optional): the same W with a box of bn / 2 rows, which the half-width units of a
// split last wave load instead of full-height tiles. With it, bf16 launches with bn = 256 (other
// than epilogue 4) run on CTA pairs: 256 x 256 tiles, each CTA of a pair loading 128 rows of A and
// bn / 2 rows of W through tmW_half (unless WENC_GEMM_PAIR=0 in the environment).
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmW, int M, int N, int K, int bn, int epilogue,
                        const float* bias, const float* resid, void* out, uint32_t* err, int num_sms,
                        cudaStream_t stream, bool tf32 = false, int row_period = 0, const GemmExtra& ex = GemmExtra(),
                        const CUtensorMap* tmW_half = nullptr);

// ---------------------------------------------------------------- attention (tcgen05)
// Q/K/V tiles are read through 3-D maps [B][T][row] (box 64 x 128 elements for all three);
// head h of Q, K, V starts at column q_col0 + 64h, k_col0 + 64h, v_col0 + 64h. A persistent grid
// (one CTA per SM) walks work items of 2 * kAttnBQ query rows of one (window, head).
// out: bf16, row (b*T + t) at out + (b*T+t)*out_stride + 64h.
// With n_splits > 1 the key tiles are divided among n_splits CTAs per query pair, which write
// unnormalised partial results to part_o [n_splits*B*H*T, 64] and (max, sum) to part_ml; a second
// kernel merges them into out. n_splits is clamped to the number of key tiles.
constexpr int kAttnBQ = 128;
constexpr int kAttnBKV = 128;
constexpr int kAttnHD = 64;
int attention_pick_splits(int B, int T, int H, int num_sms);  // 1 unless the grid would be small
size_t attention_partial_bytes(int B, int T, int H, int n_splits);
cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int q_col0,
                             int k_col0, int v_col0, uint16_t* out, int out_stride, int B, int T, int H,
                             uint32_t* err, cudaStream_t stream, int n_splits = 1, float* part_o = nullptr,
                             float2* part_ml = nullptr);
// The two launches of launch_attention, separately (for per-launch accounting).
// stop_after >= 0 (self-test only, wenc_selftest_attention_abort): the TMA producer gives up after
// that many K tiles as if one of its waits had run out; -1 everywhere else.
cudaError_t launch_attention_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int q_col0,
                                  int k_col0, int v_col0, uint16_t* out, int out_stride, int B, int T, int H,
                                  uint32_t* err, cudaStream_t stream, int n_splits, float* part_o, float2* part_ml,
                                  int stop_after = -1);
cudaError_t launch_attention_combine(const float* part_o, const float2* part_ml, uint16_t* out, int out_stride, int B,
                                     int T, int H, int n_splits, cudaStream_t stream);
int attention_launches(int T, int n_splits);  // kernels one launch_attention makes (1 or 2)

// TF32 attention: Q/K/V fp32 [B][T][row] through 3-D fp32 maps (box 32 x 128 for Q, 32 x
// kAttnTf32BKV for K and V; each 64-wide head is read as two 32-column boxes); out fp32
// rounded to TF32, row (b*T+t) at out + (b*T+t)*out_stride + 64h. A persistent grid walks work
// items of 2 x 128 queries of one (window, head).
constexpr int kAttnTf32BQ = 128;
constexpr int kAttnTf32BKV = 64;
cudaError_t launch_attention_tf32(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int q_col0,
                                  int k_col0, int v_col0, float* out, int out_stride, int B, int T, int H,
                                  uint32_t* err, cudaStream_t stream);

// ---------------------------------------------------------------- convolutional stem
// Unfold for a kernel-3, padding-1 convolution over time: x [B, t_in, C] (fp32, or the operand
// format: bf16 / TF32-rounded fp32) -> A [B * t_out, k_pad] in the operand format with
// A[b*t_out + t, j*C + i] = x[b, stride*t + j - 1, i] (0 outside the window) and zeros in
// columns 3C .. k_pad-1. C % 8 == 0, k_pad % 8 == 0, k_pad >= 3C.
cudaError_t launch_unfold3(const void* x, bool x_f32, void* a, bool a_tf32, int B, int t_in, int C, int stride,
                           int k_pad, cudaStream_t stream);
// Weight in unfold order: w [C_out, C_in, 3] (fp32 or bf16) -> wp [C_out, k_pad] in the operand
// format with wp[o, j*C_in + i] = w[o, i, j], zeros in columns 3*C_in .. k_pad-1.
cudaError_t launch_conv_weight(const void* w, bool w_bf16, void* wp, bool wp_tf32, int c_out, int c_in, int k_pad,
                               cudaStream_t stream);

// ---------------------------------------------------------------- weight packing
cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, size_t n, cudaStream_t stream);
// fp32 (rounded to TF32, nearest, ties away) or bf16 (widened, exact) -> fp32 for the TF32 path.
cudaError_t launch_to_tf32(const void* src, bool src_bf16, float* dst, size_t n, cudaStream_t stream);

}  // namespace wenc_host
