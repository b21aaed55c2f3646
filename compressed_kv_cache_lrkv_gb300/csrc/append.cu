// append.cu -- Eqs. (4)-(5) of "Low-Rank Key Value Attention": write the
// compressed cache rows of new tokens.
//
//   Y = X W_cat,  W_cat = [W_shared^K | W_shared^V | U_1^K..U_H^K | U_1^V..U_H^V]
//   s^K_t = Y[t, 0:d_h], s^V_t = Y[t, d_h:2d_h], z^K_{h,t} = Y[t, 2d_h + h r : 2d_h + (h+1) r], z^V likewise.
//
// This file holds the bandwidth-bound variant used when few rows are appended
// (a decode step appends one row per sequence): the weight rows (W_cat^T,
// contiguous along d) are streamed exactly once with 16-byte loads, for up to
// NT token rows at a time.  fp32 accumulation in a fixed order, round to
// nearest even to bf16, scatter to the row's slot.
#include "kernels.h"
#include "lrkv_internal.cuh"

namespace lrkv {


// Store one finished fp32 value of output column `col` for token slot `slot`.
__device__ __forceinline__ void store_cache_value(const AppendArgs& a, long long slot, int col, float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    const uint16_t bits = *reinterpret_cast<const uint16_t*>(&b);
    if (col < a.d_h)
        a.sK[slot * a.d_h + col] = bits;
    else if (col < 2 * a.d_h)
        a.sV[slot * a.d_h + col - a.d_h] = bits;
    else if (col < 2 * a.d_h + a.HR)
        a.zK[slot * a.HR + col - 2 * a.d_h] = bits;
    else
        a.zV[slot * a.HR + col - 2 * a.d_h - a.HR] = bits;
}

// Slot of row t, or -1 to skip it (negative entry: padding; too large: status bit).
__device__ __forceinline__ long long checked_slot(const AppendArgs& a, int t) {
    const long long s = a.slots[t];
    if (s < 0) return -1;
    if (s >= a.nslots) {
        set_status(a.status, LRKV_DEV_BAD_SLOT);
        return -1;
    }
    return s;
}

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x) {
    float acc = bf16lo(w.x) * bf16lo(x.x);
    acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
    acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc);
    acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
    acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc);
    acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
    acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc);
    acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
    return acc;
}

// One CTA owns COLS consecutive output columns; its 8 warps split the K
// (hidden) dimension -- lane l of warp w reads 16-byte chunks
// k = (w * 32 + l) * 8 + i * 2048 -- so every weight byte is read once, with
// up to COLS * ceil(d / 2048) independent 16-byte loads in flight per lane.
// Partial sums are reduced with warp shuffles and then across warps in shared
// memory, always in the same order.
template <int NT, int COLS>
__global__ void __launch_bounds__(256) append_rowwise_kernel(const AppendArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = blockIdx.x * COLS;
    const int t0 = blockIdx.y * NT;
    __shared__ float red[8][COLS * NT];
    float acc[COLS][NT];
#pragma unroll
    for (int c = 0; c < COLS; ++c)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[c][t] = 0.f;

    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll 2
    for (int k = (warp * 32 + lane) * 8; k < a.d; k += 256 * 8) {
        uint4 w[COLS];
#pragma unroll
        for (int c = 0; c < COLS; ++c)
            w[c] = (c0 + c < a.N) ? __ldg(reinterpret_cast<const uint4*>(a.W + (size_t)(c0 + c) * a.d + k)) : zero;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t0 + t < a.n) {
                const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)(t0 + t) * a.d + k));
#pragma unroll
                for (int c = 0; c < COLS; ++c) acc[c][t] += dot8(w[c], x);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < COLS; ++c)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float v = acc[c][t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) red[warp][c * NT + t] = v;
        }
    __syncthreads();
    for (int i = threadIdx.x; i < COLS * NT; i += 256) {
        const int c = i / NT, t = i % NT;
        if (c0 + c < a.N && t0 + t < a.n) {
            float v = 0.f;
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) v += red[ww][i];
            const long long slot = checked_slot(a, t0 + t);
            if (slot >= 0) store_cache_value(a, slot, c0 + c, v);
        }
    }
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
#define LRKV_ROW(NTV, COLSV)                                                             \
    {                                                                                    \
        dim3 grid((a.N + COLSV - 1) / COLSV, (a.n + NTV - 1) / NTV);                     \
        append_rowwise_kernel<NTV, COLSV><<<grid, 256, 0, stream>>>(a);                  \
        return cudaGetLastError();                                                       \
    }
    if (a.n <= 1) LRKV_ROW(1, 4)
    if (a.n <= 2) LRKV_ROW(2, 4)
    if (a.n <= 4) LRKV_ROW(4, 4)
    if (a.n <= 8) LRKV_ROW(8, 4)
    LRKV_ROW(16, 2)
#undef LRKV_ROW
}

}  // namespace lrkv
