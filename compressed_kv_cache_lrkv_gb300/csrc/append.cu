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
    const int dk = a.d_h + a.d_rope;  // shared key row: [s^K | k^R]
    if (col < dk)
        a.sK[slot * dk + col] = bits;
    else if (col < dk + a.d_h)
        a.sV[slot * a.d_h + col - dk] = bits;
    else if (col < dk + a.d_h + a.HR)
        a.zK[slot * a.HR + col - dk - a.d_h] = bits;
    else
        a.zV[slot * a.HR + col - dk - a.d_h - a.HR] = bits;
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

// Partial dot products of this thread's chunks of NCOL weight rows (w0, and w1 when NCOL == 2)
// with the block's NT hidden rows.
template <int NT, int NCOL>
__device__ __forceinline__ void rowwise_partials(const AppendArgs& a, const uint16_t* w0, const uint16_t* w1, int t0,
                                                 float (&acc)[2][NT]) {
    const int nchunk = a.d >> 3;
#pragma unroll 4
    for (int k8 = threadIdx.x; k8 < nchunk; k8 += 128) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(w0) + k8);
        uint4 w1v = make_uint4(0, 0, 0, 0);
        if (NCOL == 2) w1v = __ldg(reinterpret_cast<const uint4*>(w1) + k8);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t0 + t < a.n) {
                const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)(t0 + t) * a.d) + k8);
                acc[0][t] += dot8(w, x);
                if (NCOL == 2) acc[1][t] += dot8(w1v, x);
            }
        }
    }
}

// One 128-thread CTA per output column c and block of NT token rows: lane i of
// the CTA reads the 16-byte chunks i, i + 128, ... of weight row c (W_cat^T is
// contiguous along d), so the whole weight matrix is in flight in about one
// memory round trip (N CTAs, one wave); the NT hidden rows are small and
// stay in L1/L2.  Partial sums are reduced with warp shuffles and then across
// the four warps in shared memory, always in the same order.  In the range of the
// shared positional key a CTA computes the two columns of one rotation pair and turns
// them at each row's position before rounding.
template <int NT, bool ROPE>
__global__ void __launch_bounds__(128) append_rowwise_kernel(const AppendArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.x, half = ROPE ? a.d_rope / 2 : 0;
    const bool pair = ROPE && u >= a.d_h && u < a.d_h + half;  // uniform over the CTA
    const int c = (ROPE && u >= a.d_h) ? (pair ? a.d_h + 2 * (u - a.d_h) : u + half) : u;
    const int t0 = blockIdx.y * NT;
    __shared__ float red[ROPE ? 2 : 1][4][NT];
    float acc[2][NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[0][t] = acc[1][t] = 0.f;
    const uint16_t* wrow = a.W + (size_t)c * a.d;
    if (ROPE && pair)
        rowwise_partials<NT, 2>(a, wrow, wrow + a.d, t0, acc);
    else
        rowwise_partials<NT, 1>(a, wrow, wrow, t0, acc);
#pragma unroll
    for (int j = 0; j < (ROPE ? 2 : 1); ++j)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float v = acc[j][t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) red[j][warp][t] = v;
        }
    __syncthreads();
    if (threadIdx.x < NT && t0 + threadIdx.x < a.n) {
        const int t = threadIdx.x;
        float v0 = (red[0][0][t] + red[0][1][t]) + (red[0][2][t] + red[0][3][t]);
        const long long slot = checked_slot(a, t0 + t);
        if (slot >= 0) {
            if (ROPE && pair) {
                float v1 = (red[ROPE ? 1 : 0][0][t] + red[ROPE ? 1 : 0][1][t]) +
                           (red[ROPE ? 1 : 0][2][t] + red[ROPE ? 1 : 0][3][t]);
                rope_pair(v0, v1, u - a.d_h, a.d_rope, a.positions[t0 + t], a.rope_base);
                store_cache_value(a, slot, c + 1, v1);
            }
            store_cache_value(a, slot, c, v0);
        }
    }
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
#define LRKV_ROW(NTV)                                                                    \
    {                                                                                    \
        dim3 grid(a.N - a.d_rope / 2, (a.n + NTV - 1) / NTV); /* pairs: one CTA each */ \
        if (a.d_rope > 0)                                                                \
            append_rowwise_kernel<NTV, true><<<grid, 128, 0, stream>>>(a);               \
        else                                                                             \
            append_rowwise_kernel<NTV, false><<<grid, 128, 0, stream>>>(a);              \
        return cudaGetLastError();                                                       \
    }
    if (a.n <= 1) LRKV_ROW(1)
    if (a.n <= 2) LRKV_ROW(2)
    if (a.n <= 4) LRKV_ROW(4)
    if (a.n <= 8) LRKV_ROW(8)
    LRKV_ROW(16)
#undef LRKV_ROW
}

}  // namespace lrkv
