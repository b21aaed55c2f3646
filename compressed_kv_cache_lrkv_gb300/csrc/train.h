// train.h -- internal interface of the training-time projection kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lrkv {

// C = A . B on the tensor cores (bf16 operands, fp32 accumulation), 128 x BN output tiles
// (BN = 64, 128, 160 or 256), batched over nbatch * ksplit.  Operand boxes are read through 2-D
// tensor maps (128-byte swizzle): a K-major operand is a [rows][K] map read in 64-wide boxes of
// 128 (A) or BN (B) rows, an MN-major one a [K][rows] map read in 64 x 64 boxes.  Coordinates of batch z start at
// (x0 + z * zx, y0 + z * zy).  With kfix > 0 (K-major operands only) the first kfix K columns
// are shared by all batches: A's come from columns [0, kfix) of its map and B's from a second map
// at (k, n0); K column k >= kfix is column k - kfix of the batch's own operand boxes.  Output:
// bf16, or for split-K partials fp32 at C + ((batch * ksplit + ks) * 128 + row) * BN.  With
// tma_out the bf16 tile goes out through shared memory by TMA stores of a 3-D map {N, nbatch, M}
// (strides c_zstride and ldc; 32 x 1 x 32 boxes, 64-byte swizzle).
struct GemmArgs {
    void* C;
    int ldc;                  // elements
    long long c_zstride;      // elements between batches (bf16 output)
    int M, N, K;              // rows and columns stored, contraction length
    int a_x0, a_y0, a_zx, a_zy;
    int b_x0, b_y0, b_zx, b_zy;
    int nbatch, ksplit;
    int kfix;                 // leading K columns shared by all batches (multiple of 64)
    int a_mn, b_mn;           // operand is MN-major ([K][rows] map) rather than K-major
    int tma_out;              // 1: store through the output map
    uint32_t* status;
};

// Operand and output maps and arguments of up to two products run by one launch (their tiles
// concatenated, group 0 first); B2 is the second B map of group 0 (kfix).
struct TGemmParams {
    CUtensorMap A[2], B[2], C[2], B2;
    GemmArgs g[2];
    int ngroups;
    int tiles0, total;  // tiles of group 0, of all groups
    int* ctr;           // work queue (zero at launch) or null: round-robin tiles
};

// Launch C = A . B with 128 x bn tiles (operand majors in g.a_mn / g.b_mn); out_f32: fp32 split-K
// partials.  Tile widths: expansion and dR 128, Y 160, dW_T and dX 256, dB partials 64 (fp32).
cudaError_t launch_tgemm(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tB2, const CUtensorMap& tC,
                         const GemmArgs& g, int bn, bool out_f32, cudaStream_t stream);

// Two bf16-output products in one launch whose CTAs take tiles from a shared queue (`ctr`, one int
// of device memory, zeroed here first): group 0's tiles are handed out first.
cudaError_t launch_tgemm2(const CUtensorMap* tA, const CUtensorMap* tB, const CUtensorMap* tC, const GemmArgs* g, int bn,
                          int* ctr, cudaStream_t stream);

// Device address of a 128 x 128 bf16 identity matrix (row-major), or null.
const void* train_identity();

// Fused pass over dK for 128-token tiles: G = sum_h dK_h into Gc columns [0, d_h) and dR_h =
// dK_h B_h into Gc columns d_h + h r .., each dK_h tile read once (a CTA pair splits the heads).
struct DkArgs {
    uint16_t* Gc;
    int ldg;                  // Gc row pitch, elements
    int n, H, d_h, r;
    float* dBp;               // fp32 dB partials [H][n / 128 tiles][d_h][r], or null (dB not folded in)
    int rx0;                  // column of R_1 in the map tR (d_h)
    uint32_t* status;
};
bool dk_pass_supported(int H, int d_h, int r);
bool dk_pass_folds_dB(int H, int d_h, int r);
// tdK: [n][H d_h] in 64 x 128 boxes; tBT: BT = [H r][d_h] in 64 x r boxes, written here from the
// residual factors B [H][d_h][r] first; tR (with dBp): Y = [S | R] in 16 x 128 boxes (32-byte swizzle).
cudaError_t launch_dk_pass(const CUtensorMap& tdK, const CUtensorMap& tBT, const CUtensorMap& tR, const uint16_t* B,
                           uint16_t* BT, const DkArgs& a, cudaStream_t stream);

// G[t] = sum_h dK[t][h][:] into columns [0, d_h) of Gc [n][ldg] (bf16, fp32 sums).
cudaError_t launch_head_sum(const uint16_t* dK, uint16_t* Gc, int n, int H, int d_h, int ldg, cudaStream_t stream);

// dB[h][e][j] = sum over split-K partials P[h][ks][e][0..pw) (in ks order), j < r, bf16.
cudaError_t launch_dB_reduce(const float* P, uint16_t* dB, int H, int ksplit, int d_h, int r, int pw,
                             cudaStream_t stream);

}  // namespace lrkv
