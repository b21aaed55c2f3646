// train.h -- internal interface of the training-time projection kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lrkv {

// C = A . B on the tensor cores (bf16 operands, fp32 accumulation), 128 x 128 output tiles,
// batched over grid.z = nbatch * ksplit.  Operand boxes are read through 2-D tensor maps
// (128-byte swizzle): a K-major operand is a [rows][K] map read in 64 x 128 boxes, an MN-major
// one a [K][rows] map read in two 64 x 64 boxes per stage.  Coordinates of batch z start at
// (x0 + z * zx, y0 + z * zy).  Output: bf16 (optionally plus a bf16 matrix `add`, rounded
// once) or, for split-K partials, fp32 at C + ((batch * ksplit + ks) * M_pad) * ldc.
struct GemmArgs {
    void* C;
    int ldc;                  // elements
    long long c_zstride;      // elements between batches (bf16 output)
    int M, N, K;              // rows and columns stored, contraction length
    int a_x0, a_y0, a_zx, a_zy;
    int b_x0, b_y0, b_zx, b_zy;
    int nbatch, ksplit;
    const uint16_t* add;      // bf16 matrix added in the epilogue (or null)
    int ld_add;
    uint32_t* status;
};

// Launch C = A . B.  AMN / BMN: operand is MN-major; OUTF32: fp32 split-K partials.
cudaError_t launch_tgemm(const CUtensorMap& tA, const CUtensorMap& tB, const GemmArgs& g, bool a_mn, bool b_mn,
                         bool out_f32, cudaStream_t stream);

// G[t] = sum_h dK[t][h][:] into columns [0, d_h) of Gc [n][ldg] (bf16, fp32 sums).
cudaError_t launch_head_sum(const uint16_t* dK, uint16_t* Gc, int n, int H, int d_h, int ldg, cudaStream_t stream);

// dB[h][e][j] = sum over split-K partials P[h][ks][e][0..127] (in ks order), j < r, bf16.
cudaError_t launch_dB_reduce(const float* P, uint16_t* dB, int H, int ksplit, int d_h, int r, cudaStream_t stream);

}  // namespace lrkv
