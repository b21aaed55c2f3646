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
// nearest even to bf16 (after rotating the positional-key pairs), scatter to
// the row's slot.
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

constexpr int kSplitCols = 64;   // output columns per CTA: 8 warps x 8 columns, 4 lanes per column

// Few-row append (a decode step appends one row per sequence): a GEMV-like stream of W_cat^T.
// A cluster of KS CTAs shares a group of 64 output columns and splits d into KS slices: each CTA
// holds its slice of the NT hidden rows in shared memory and streams its slice of the 64 weight
// rows once (16-byte loads, 4 lanes per row covering 64 contiguous bytes per step), so the hidden
// rows are read KS * (N / 64) times in all instead of once per output column.  The fp32 partial
// sums are reduced across the cluster through distributed shared memory by rank 0 in rank order
// (deterministic), which then rounds (after rotating the positional-key pairs) and stores.
template <int NT, bool ROPE>
__global__ void __launch_bounds__(256) append_splitk_kernel(const AppendArgs a, int kslice) {
    extern __shared__ __align__(16) uint8_t xs_raw[];
    __shared__ float part[NT][kSplitCols];
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(xs_raw);  // [NT][kslice]
    const uint32_t r = cluster_ctarank(), KS = cluster_nctarank();
    const int group = blockIdx.x / KS;
    const int t0 = blockIdx.y * NT;
    const int k0 = (int)r * kslice, k1 = min(a.d, k0 + kslice);
    const int nk8 = kslice >> 3;  // 16-byte chunks per hidden-row slice
    for (int idx = threadIdx.x; idx < NT * nk8; idx += blockDim.x) {
        const int t = idx / nk8, c8 = idx - t * nk8;
        const int k = k0 + c8 * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t0 + t < a.n && k < k1) v = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)(t0 + t) * a.d + k));
        reinterpret_cast<uint4*>(xs_raw)[idx] = v;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cl = warp * 8 + (lane >> 2), q = lane & 3;
    const int col = group * kSplitCols + cl;
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    if (col < a.N) {
        const uint16_t* wrow = a.W + (size_t)col * a.d;
#pragma unroll 4
        for (int k = k0 + q * 8; k < k1; k += 32) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(wrow + k));
            const int c8 = (k - k0) >> 3;
#pragma unroll
            for (int t = 0; t < NT; ++t)
                acc[t] += dot8(w, reinterpret_cast<const uint4*>(xs)[t * nk8 + c8]);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 1);
        acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 2);
    }
    if (q == 0)
#pragma unroll
        for (int t = 0; t < NT; ++t) part[t][cl] = acc[t];
    cluster_sync_all();
    if (r == 0) {
        // (row, column) pairs spread over all threads; each thread's KS partials are loaded
        // together and summed in rank order.  Columns c and c ^ 1 sit in adjacent lanes.
        for (int pidx = threadIdx.x; pidx < NT * kSplitCols; pidx += blockDim.x) {
            const int t = pidx / kSplitCols, cc = pidx % kSplitCols;
            const int c = group * kSplitCols + cc;
            const uint32_t src = (uint32_t)__cvta_generic_to_shared(&part[t][cc]);
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
                    rope_pair(x0, x1, (c - a.d_h) >> 1, a.d_rope, a.positions[t0 + t], a.rope_base);
                    v = (cc & 1) ? x1 : x0;
                }
            }
            if (slot >= 0 && c < a.N) store_cache_value(a, slot, c, v);
        }
    }
    cluster_sync_all();  // rank 0 has read every CTA's partials before any of them exits
}

template <int NT, bool ROPE>
static cudaError_t launch_splitk(const AppendArgs& a, int ks, int kslice, cudaStream_t stream) {
    auto kern = append_splitk_kernel<NT, ROPE>;
    const size_t smem = (size_t)NT * kslice * 2;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(((a.N + kSplitCols - 1) / kSplitCols) * ks, (a.n + NT - 1) / NT);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, kslice);
}

static cudaError_t launch_rowwise(const AppendArgs& a, cudaStream_t stream) {
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

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    // Weight streams up to 64 MB: one CTA per output column (the hidden rows stay in L1/L2 at that
    // size and there is no cluster setup); larger ones re-read the hidden rows once per column
    // from L2, so they go through the split-K cluster kernel below.
    if ((long long)a.N * a.d * 2 < (64LL << 20)) return launch_rowwise(a, stream);
    // Split d so that the grid has about two CTAs per SM (at most 8 per cluster, slices of at
    // least 32 elements), so the weight stream keeps every SM's loads in flight.
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int groups = (a.N + kSplitCols - 1) / kSplitCols;
    int nt = a.n <= 1 ? 1 : a.n <= 2 ? 2 : a.n <= 4 ? 4 : a.n <= 8 ? 8 : 16;
    const int rowblocks = (a.n + nt - 1) / nt;
    int ks = (2 * sms + groups * rowblocks - 1) / (groups * rowblocks);
    ks = ks < 1 ? 1 : ks > 8 ? 8 : ks;
    // the hidden-row slice (nt rows x d / ks) must fit in shared memory: more slices, then fewer rows
    const long long kMaxSlice = 192 * 1024;
    while (ks < 8 && (long long)nt * ((a.d + ks - 1) / ks) * 2 > kMaxSlice) ++ks;
    while (ks > 1 && (a.d + ks - 1) / ks < 32) --ks;
    const int kslice = (((a.d + ks - 1) / ks) + 31) & ~31;
    while (nt > 1 && (long long)nt * kslice * 2 > kMaxSlice) nt >>= 1;
    if ((long long)nt * kslice * 2 > kMaxSlice) return cudaErrorInvalidValue;
#define LRKV_SPLITK(NTV)                                                                        \
    if (nt == NTV)                                                                              \
        return a.d_rope > 0 ? launch_splitk<NTV, true>(a, ks, kslice, stream)                    \
                            : launch_splitk<NTV, false>(a, ks, kslice, stream);
    LRKV_SPLITK(1) LRKV_SPLITK(2) LRKV_SPLITK(4) LRKV_SPLITK(8) LRKV_SPLITK(16)
#undef LRKV_SPLITK
    return cudaErrorInvalidValue;
}

}  // namespace lrkv
