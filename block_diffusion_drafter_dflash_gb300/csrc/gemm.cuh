// GEMM launch interface shared by the host orchestration and the kernels.
#pragma once

#include "common.cuh"
#include "epilogue.cuh"

namespace dflash {

// How one GEMM launch is cut: token rows per CTA tile, split-K.
struct GemmPlan {
  int tc;               // 1: tcgen05 tensor-core kernel, 0: CUDA-core kernel
  int planes;           // activation planes the kernel reads
  int bm;               // token rows per CTA tile
  int token_tiles;
  int splits;
  int kblocks_per_split;  // 64-column blocks of K per split
  int stages;             // pipeline depth of the tensor-core kernel
  size_t smem;            // dynamic shared memory per CTA
  size_t partial_floats;  // split-K scratch floats (0 if splits == 1)
  int counters;           // split-K tile counters (0 if splits == 1)
  int dense;              // persistent many-row kernel: `grid` CTAs walk all tiles, no split-K
  int grid;
};

// Decide the cut for an M x (tiles*128) x K product on a device with `sms` SMs.
// bf16 products use the tcgen05 kernel unless `tc` is 0.
// `planes` = activation planes (2 for a hi/lo bf16 pair).
GemmPlan plan_gemm(int dtype, int M, int K, int tiles, int sms, int tc, int planes);
GemmPlan plan_gemm_tc(int M, int K, int tiles, int sms, int planes);
size_t dense_smem(int stages);   // shared memory of the persistent many-row kernel

// Tensor maps (CUtensorMap, 128 B each) for the tensor-core kernels: a weight
// matrix [rows][inner] bf16 read in 64 x box_rows boxes (64 for the GEMM
// kernel, 128 for the persistent one), and an activation matrix
// [rows][row_stride] bf16 read in 64 x box_rows boxes.  128-byte swizzle.
bool encode_weight_map(void* map, const void* base, int inner, int rows, int box_rows = kHalfN);
bool encode_activation_map(void* map, const void* base, int inner, int rows, int row_stride, int box_rows);
size_t tensor_map_bytes();

template <class Epi>
cudaError_t gemm_tc_launch(const GemmProblem& p, const GemmPlan& plan, const Epi& epi, cudaStream_t s);

// Fill the plan's fields into the problem (splits, kblocks, scratch pointers).
void apply_plan(GemmProblem& p, const GemmPlan& plan, float* partial, int* counters);

template <typename T, class Epi>
cudaError_t gemm_launch(const GemmProblem& p, const GemmPlan& plan, const Epi& epi, cudaStream_t s);

}  // namespace dflash
