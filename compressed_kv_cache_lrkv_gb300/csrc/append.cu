// append.cu -- Eqs. (4)-(5) of "Low-Rank Key Value Attention": write the
// compressed cache rows of new tokens.
//
//   Y = X W_cat,  W_cat = [W_shared^K | W_shared^V | U_1^K..U_H^K | U_1^V..U_H^V]
//   s^K_t = Y[t, 0:d_h], s^V_t = Y[t, d_h:2d_h], z^K_{h,t} = Y[t, 2d_h + h r : 2d_h + (h+1) r], z^V likewise.
//
// This file holds the bandwidth-bound variants used when few rows are appended
// (a decode step appends one row per sequence): the weight rows (W_cat^T,
// contiguous along d) are streamed exactly once with 16-byte loads, for a block
// of token rows at a time -- on the CUDA cores a warp per column for d <= 1024
// and a CTA per column below 64 MB of weights, as a split-K product on the
// warp-level tensor cores above.  A layer-batched call runs every layer in the
// same launch (grid z = layer, per-layer strides in the arguments).  fp32
// accumulation in a fixed order, round to nearest even to bf16 (after rotating
// the positional-key pairs), scatter to the row's slot.
#include "kernels.h"
#include "lrkv_internal.cuh"
#include "rotary.cuh"

namespace lrkv {


// The arguments of layer z of a layer-batched launch (z = 0 or a single layer: unchanged).
__device__ __forceinline__ AppendArgs layer_args(const AppendArgs& a, int z) {
    AppendArgs l = a;
    l.X += z * a.ls_X;
    l.W += z * a.ls_W;
    l.sK += z * a.ls_sK;
    l.sV += z * a.ls_sV;
    l.zK += z * a.ls_zK;
    l.zV += z * a.ls_zV;
    return l;
}

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
    // Rows past n read the last row instead (their sums are never stored), so that every load
    // of a chunk is issued before the first is used.
    const uint4* xr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) xr[t] = reinterpret_cast<const uint4*>(a.X + (size_t)min(t0 + t, a.n - 1) * a.d);
#pragma unroll 2
    for (int k8 = threadIdx.x; k8 < nchunk; k8 += 128) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(w0) + k8);
        uint4 w1v = make_uint4(0, 0, 0, 0);
        if (NCOL == 2) w1v = __ldg(reinterpret_cast<const uint4*>(w1) + k8);
        uint4 x[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) x[t] = __ldg(xr[t] + k8);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[0][t] += dot8(w, x[t]);
            if (NCOL == 2) acc[1][t] += dot8(w1v, x[t]);
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
__global__ void __launch_bounds__(128) append_rowwise_kernel(const AppendArgs a0) {
    const AppendArgs a = layer_args(a0, blockIdx.z);
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
                rope_rotate(v0, v1, u - a.d_h, a.d_rope, a.positions[t0 + t], a.rope_base);
                store_cache_value(a, slot, c + 1, v1);
            }
            store_cache_value(a, slot, c, v0);
        }
    }
}

// Few rows and a small hidden size (d <= 1024): one warp per output column, or per rotation pair
// of the positional key (8 warps per CTA).  Lane l sums the 16-byte chunks l, l + 32, ... of the
// column's weight row with the block's NT hidden rows (small, shared by every warp: L1 / L2
// hits).  The V = NCOL x NT partial sums are then reduced across the warp by recursive halving:
// at the step with lane mask m, a lane keeps one half of its values, adds the partner's copy of
// that half and hands over the other half, so after log2(V) steps lane l holds value
// (l >> (5 - log2 V)) summed over 2^log2(V) lanes, and the remaining masks finish the sum
// (log2 V + ... shuffles instead of 5 V).  The order of the additions is fixed.
template <int NT, bool ROPE>
__global__ void __launch_bounds__(256) append_warp_kernel(const AppendArgs a0) {
    const AppendArgs a = layer_args(a0, blockIdx.z);
    constexpr int NCOL = ROPE ? 2 : 1;
    constexpr int V = NCOL * NT;                                // values per lane: [column][row]
    constexpr int LOGV = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : V >= 2 ? 1 : 0;
    static_assert((1 << LOGV) == V, "V is a power of two <= 32");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = ROPE ? a.d_rope / 2 : 0;
    const int u = blockIdx.x * 8 + warp;
    if (u >= a.N - half) return;  // (warp-uniform; the kernel has no block-wide barrier)
    const bool pair = ROPE && u >= a.d_h && u < a.d_h + half;
    const int c = (ROPE && u >= a.d_h) ? (pair ? a.d_h + 2 * (u - a.d_h) : u + half) : u;
    const int t0 = blockIdx.y * NT;
    float v[V];
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] = 0.f;
    const uint4* w0 = reinterpret_cast<const uint4*>(a.W + (size_t)c * a.d);
    const uint4* w1 = reinterpret_cast<const uint4*>(a.W + (size_t)(c + 1) * a.d);
    const int nchunk = a.d >> 3;
    // Rows past n read the last row instead (their sums are never stored), so that every load
    // of a chunk is issued before the first is used.
    const uint4* xr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) xr[t] = reinterpret_cast<const uint4*>(a.X + (size_t)min(t0 + t, a.n - 1) * a.d);
    for (int k8 = lane; k8 < nchunk; k8 += 32) {
        const uint4 w = __ldg(w0 + k8);
        uint4 wb = make_uint4(0, 0, 0, 0);
        if (ROPE && pair) wb = __ldg(w1 + k8);
        uint4 x[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) x[t] = __ldg(xr[t] + k8);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            v[t] += dot8(w, x[t]);
            if (ROPE) v[NT + t] += dot8(wb, x[t]);
        }
    }
    // recursive halving over masks 16, 8, ..., then plain butterflies
#pragma unroll
    for (int step = 0, n = V; step < 5; ++step) {
        const int m = 16 >> step;
        if (n > 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < n / 2) {
                    const float keep = upper ? v[i + n / 2] : v[i];
                    const float give = upper ? v[i] : v[i + n / 2];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, m);
                }
            }
            n >>= 1;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
        }
    }
    const int vi = LOGV == 0 ? 0 : (lane >> (5 - LOGV)) & (V - 1);
    const int col = vi / NT, t = vi - (vi / NT) * NT;
    float other = 0.f;
    if (ROPE) other = __shfl_xor_sync(0xffffffffu, v[0], 16);  // the pair's other column, same row
    const bool writer = (lane & ((32 >> LOGV) - 1)) == 0 && col == 0 && t0 + t < a.n;
    if (writer) {
        const long long slot = checked_slot(a, t0 + t);
        if (slot >= 0) {
            float x0 = v[0];
            if (ROPE && pair) {
                float x1 = other;
                rope_rotate(x0, x1, u - a.d_h, a.d_rope, a.positions[t0 + t], a.rope_base);
                store_cache_value(a, slot, c + 1, x1);
            }
            store_cache_value(a, slot, c, x0);
        }
    }
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Load a float from the shared memory of CTA `rank` of this cluster (no ordering constraint:
// the caller has passed a cluster barrier since the value was written).
__device__ __forceinline__ float ld_cluster_f32(uint32_t local, uint32_t rank) {
    uint32_t ra;
    float v;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra));
    return v;
}

// 16-byte load of streamed data that is read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_16(const uint16_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

constexpr int kMmaCols = 32;         // output columns per CTA: two 16-row tiles of W_cat^T
constexpr int kMmaPitch = kMmaCols + 4;  // partial-sum row pitch in floats (conflict-free stores)

// Few-row append on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulation):
// C[col][t] = sum_k W_cat^T[col][k] X[t][k], with the weight columns on M and the 8 (NB = 1) or
// 16 (NB = 2) token rows of the CTA on N.  The order in which k enters an MMA is free (a sum), so
// every operand fragment is loaded straight from global memory as one 16-byte group per thread
// and row: lane (g, q) of a warp reads elements [k + 8q, k + 8q + 8) of weight rows g and g + 8 of
// each 16-row tile and of token row g, and its four 32-bit words feed two MMAs (words 0 and 1 the
// first, 2 and 3 the second) as the pairs the fragment layout assigns to that lane; the A and B
// operands see the same permutation of k.  No shared-memory staging: the weight stream (read once)
// goes from HBM to registers, one 64-wide k step ahead of the MMAs.
//
// Work split: a cluster of KS CTAs owns 32 output columns and one block of token rows; each of
// the 8 warps of each CTA sums a contiguous range of kwarp elements of k.  The warps' fp32 partial
// sums are combined in shared memory in warp order, and the CTAs' through distributed shared
// memory by rank 0 in rank order (deterministic), which then rounds (after rotating the
// positional-key pairs) and stores.
template <int NB, bool ROPE>
__global__ void __launch_bounds__(256, 2) append_mma_kernel(const AppendArgs a0, int kwarp) {
    const AppendArgs a = layer_args(a0, blockIdx.z);
    constexpr int NT = 8 * NB;
    __shared__ float part[8][NT][kMmaPitch];
    __shared__ float csum[NT][kMmaCols];
    const uint32_t r = cluster_ctarank(), KS = cluster_nctarank();
    const int group = blockIdx.x / KS;
    const int t0 = blockIdx.y * NT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int col0 = group * kMmaCols;

    // operand rows (indices clamped into range: those lanes' results are never stored)
    const uint16_t* wr[2][2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) wr[i][h] = a.W + (size_t)min(col0 + 16 * i + 8 * h + g, a.N - 1) * a.d;
    const uint16_t* xr[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) xr[j] = a.X + (size_t)min(t0 + 8 * j + g, a.n - 1) * a.d;

    float acc[NB][2][4];
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][i][e] = 0.f;

    const int kbeg = ((int)r * 8 + warp) * kwarp;
    const int kend = min(a.d, kbeg + kwarp);
    // one 64-wide step: two 32-wide halves c, lane q holding elements [k + 32c + 8q, +8)
    uint4 w[2][2][2], x[NB][2];  // w[tile][row half][c], x[row block][c]
    auto load = [&](int k, uint4 (&wv)[2][2][2], uint4 (&xv)[NB][2]) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int kk = k + 32 * c + 8 * q;
            const bool ok = kk < kend;  // d and kend are multiples of 8
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h) wv[i][h][c] = ok ? ld_stream_16(wr[i][h] + kk) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < NB; ++j)
                xv[j][c] = ok ? __ldg(reinterpret_cast<const uint4*>(xr[j] + kk)) : make_uint4(0, 0, 0, 0);
        }
    };
    if (kbeg < kend) load(kbeg, w, x);
    for (int k = kbeg; k < kend; k += 64) {
        uint4 wn[2][2][2], xn[NB][2];
        if (k + 64 < kend) load(k + 64, wn, xn);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t* w0 = reinterpret_cast<const uint32_t*>(&w[i][0][c]);
                    const uint32_t* w1 = reinterpret_cast<const uint32_t*>(&w[i][1][c]);
                    const uint32_t af[4] = {w0[2 * s], w1[2 * s], w0[2 * s + 1], w1[2 * s + 1]};
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        const uint32_t* xw = reinterpret_cast<const uint32_t*>(&x[j][c]);
                        mma_16816(acc[j][i], af, xw[2 * s], xw[2 * s + 1]);
                    }
                }
        if (k + 64 < kend) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int h = 0; h < 2; ++h) w[i][h][c] = wn[i][h][c];
#pragma unroll
                for (int j = 0; j < NB; ++j) x[j][c] = xn[j][c];
            }
        }
    }
    // accumulator (j, i, e): column 16 i + g + 8 (e >> 1), token row 8 j + 2 q + (e & 1)
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[warp][8 * j + 2 * q + (e & 1)][16 * i + g + 8 * (e >> 1)] = acc[j][i][e];
    __syncthreads();
    for (int idx = threadIdx.x; idx < NT * kMmaCols; idx += blockDim.x) {
        const int t = idx / kMmaCols, cc = idx % kMmaCols;
        float v = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) v += part[ww][t][cc];
        csum[t][cc] = v;
    }
    cluster_sync_all();
    if (r == 0) {
        // (row, column) pairs spread over all threads (NT * 32 is a multiple of the block size, so
        // every lane takes part in each shuffle); columns c and c ^ 1 sit in adjacent lanes.
        for (int pidx = threadIdx.x; pidx < NT * kMmaCols; pidx += blockDim.x) {
            const int t = pidx / kMmaCols, cc = pidx % kMmaCols;
            const int c = col0 + cc;
            const uint32_t src = (uint32_t)__cvta_generic_to_shared(&csum[t][cc]);
            float pv[8];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) pv[rr] = rr < (int)KS ? ld_cluster_f32(src, rr) : 0.f;
            float v = 0.f;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
                if (rr < (int)KS) v += pv[rr];
            const long long slot = (t0 + t < a.n) ? checked_slot(a, t0 + t) : -1;
            if (ROPE) {
                // pair (2i, 2i+1) of the positional key
                const float other = __shfl_xor_sync(0xffffffffu, v, 1);
                if (c >= a.d_h && c < a.d_h + a.d_rope && slot >= 0) {
                    float x0 = (cc & 1) ? other : v, x1 = (cc & 1) ? v : other;
                    rope_rotate(x0, x1, (c - a.d_h) >> 1, a.d_rope, a.positions[t0 + t], a.rope_base);
                    v = (cc & 1) ? x1 : x0;
                }
            }
            if (slot >= 0 && c < a.N) store_cache_value(a, slot, c, v);
        }
    }
    cluster_sync_all();  // rank 0 has read every CTA's partials before any of them exits
}

template <int NB, bool ROPE>
static cudaError_t launch_mma(const AppendArgs& a, int ks, int kwarp, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(((a.N + kMmaCols - 1) / kMmaCols) * ks, (a.n + 8 * NB - 1) / (8 * NB), a.layers > 1 ? a.layers : 1);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_mma_kernel<NB, ROPE>, a, kwarp);
}

static cudaError_t launch_rowwise(const AppendArgs& a, cudaStream_t stream) {
#define LRKV_ROW(NTV)                                                                    \
    {                                                                                    \
        dim3 grid(a.N - a.d_rope / 2, (a.n + NTV - 1) / NTV, a.layers > 1 ? a.layers : 1);  \
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

static cudaError_t launch_warp(const AppendArgs& a, cudaStream_t stream) {
#define LRKV_WARP(NTV)                                                                                     \
    {                                                                                                      \
        dim3 grid((a.N - a.d_rope / 2 + 7) / 8, (a.n + NTV - 1) / NTV, a.layers > 1 ? a.layers : 1);       \
        if (a.d_rope > 0)                                                                                  \
            append_warp_kernel<NTV, true><<<grid, 256, 0, stream>>>(a);                                    \
        else                                                                                               \
            append_warp_kernel<NTV, false><<<grid, 256, 0, stream>>>(a);                                   \
        return cudaGetLastError();                                                                         \
    }
    if (a.n <= 1) LRKV_WARP(1)
    if (a.n <= 2) LRKV_WARP(2)
    if (a.n <= 4) LRKV_WARP(4)
    if (a.n <= 8) LRKV_WARP(8)
    LRKV_WARP(16)
#undef LRKV_WARP
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    // Small hidden sizes: a warp per column (a CTA per column would leave most of its threads
    // without a chunk of the row and run many small CTAs).
    if (a.d <= 1024) return launch_warp(a, stream);
    // Weight streams up to 64 MB: one CTA per output column (the hidden rows stay in L1/L2 at that
    // size and there is no cluster setup); larger ones re-read the hidden rows once per column
    // from L2, so they go through the split-K tensor-core kernel above.
    // (pairs of the positional key: one CTA each; several layers: one grid slice each)
    if ((long long)a.N * a.d * 2 < (64LL << 20)) return launch_rowwise(a, stream);
    // Split d so that the grid fills two CTAs per SM in one wave (at most 8 CTAs per cluster,
    // at least one 64-wide step per warp).
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int nb = a.n <= 8 ? 1 : 2;
    const int groups = (a.N + kMmaCols - 1) / kMmaCols;
    const int rowblocks = (a.n + 8 * nb - 1) / (8 * nb);
    const int steps = (a.d + 63) / 64;  // 64-wide k steps
    int ks = (2 * sms) / (groups * rowblocks * (a.layers > 1 ? a.layers : 1));
    ks = ks < 1 ? 1 : ks > 8 ? 8 : ks;
    while (ks > 1 && ks * 8 > steps) --ks;
    const int kwarp = ((steps + ks * 8 - 1) / (ks * 8)) * 64;
    if (a.d_rope > 0)
        return nb == 1 ? launch_mma<1, true>(a, ks, kwarp, stream) : launch_mma<2, true>(a, ks, kwarp, stream);
    return nb == 1 ? launch_mma<1, false>(a, ks, kwarp, stream) : launch_mma<2, false>(a, ks, kwarp, stream);
}

}  // namespace lrkv
