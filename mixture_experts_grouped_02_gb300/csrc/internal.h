// internal.h -- declarations shared by the library's translation units
// (kernel launchers and the C ABI in moe_abi.cu).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/moe.h"

namespace moe {

// Default wall-clock limit of any single pipeline wait inside a kernel.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// The grouped GEMMs tile 128 sorted rows (tokens) per block: the align
// block size equals the GEMM's M tile.
constexpr int kBlockM = 128;

struct AlignArgs {
  const int32_t* ids;
  int n_assign;  // T*K
  int E;
  int block_m;
  long long cap;
  int32_t* counts;
  int32_t* offsets;
  int32_t* padded_offsets;
  int32_t* sorted_ids;
  int32_t* inv_perm;
  int32_t* block_info;
  int32_t* num_blocks;
  int32_t* status;
};

// Arguments of one grouped-GEMM launch (both GEMMs).
struct GemmArgs {
  int T, H, I, E, K;
  int n_tiles;   // tiles along the output (N) dimension
  int k_tiles;   // 128-byte k-tiles over the whole reduction
  int splits;    // reduction splits (down projection); 1 for gate/up
  int band;      // N tiles per raster band
  long long cap; // rows of the padded sorted list
  const void* x;               // gate/up: token rows (T, H), gathered by cp.async
  const int32_t* sorted_ids;
  const int32_t* block_info;
  const int32_t* num_blocks;
  const float* topk_weights;  // down projection: routing weight per flat index
  void* out;                  // gate/up: h (cap, I); down: y (splits, cap, H) fp32
  int32_t* status;
  unsigned long long timeout_ns;
};

// Arguments of one block-scaled (fp8 activations x mxfp4 weights) grouped
// GEMM launch.  The reduction dimension is Kdim = H (gate/up) or I (down).
struct MxArgs {
  int T, H, I, E, K;
  int Kdim;
  int n_tiles, k_tiles, splits, band;
  long long cap;
  const uint8_t* a;            // gate/up: xq (T, H) e4m3; down: hq (cap, I) e4m3
  const float* x_row_scale;    // gate/up: per-token fp32 scale of xq
  const uint8_t* w;            // packed e2m1: w13 (E, 2I, H/2) or w2 (E, H, I/2)
  const uint8_t* w_scale;      // e8m0: (E, 2I, H/32) or (E, H, I/32)
  const int32_t* sorted_ids;
  const int32_t* block_info;
  const int32_t* num_blocks;
  const float* topk_weights;   // down: routing weight per flat index
  void* out;                   // gate/up: hq (cap, I) e4m3; down: y (splits, cap, H) fp32
  float h_scale;               // hq = e4m3(a / h_scale)
  int32_t* status;
  unsigned long long timeout_ns;
};

cudaError_t launch_mx_gate_up(const MxArgs& a, int grid, cudaStream_t s);
cudaError_t launch_mx_down(const MxArgs& a, int grid, cudaStream_t s);

cudaError_t launch_align(const AlignArgs& a, cudaStream_t s);
cudaError_t launch_combine(const float* y, int splits, long long cap, const int32_t* inv_perm,
                           int T, int K, int H, int out_dtype, void* out, int32_t* status,
                           cudaStream_t s);
cudaError_t launch_quantize_x(const void* x, int x_dtype, int T, int H, uint8_t* xq,
                              float* row_scale, cudaStream_t s);

// dtype: MOE_BF16 or MOE_F32.  tmA: down -> h (box 128 rows; unused by
// gate/up, which gathers x itself).  tmB: w13 (box 128 rows) / w2 (box 256 rows).
cudaError_t launch_gemm_gate_up(int dtype, const GemmArgs& a, const CUtensorMap& tmA,
                                const CUtensorMap& tmB, int grid, cudaStream_t s);
cudaError_t launch_gemm_down(int dtype, const GemmArgs& a, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, int grid, cudaStream_t s);

}  // namespace moe
