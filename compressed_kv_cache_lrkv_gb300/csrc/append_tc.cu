// append_tc.cu -- tensor-core path of lrkv_append for many rows (prefill chunks,
// cache builds): Y = X W_cat on the 5th-generation tensor cores, epilogue
// straight into the paged cache ("Low-Rank Key Value Attention", Eqs. (4)-(5)).
//
// One CTA computes a 128 x BN tile of Y:
//   warp 0      TMA producer: X and W_cat^T tiles (64-wide K slices, 128-byte
//               swizzle) into a 4-stage shared-memory ring;
//   warp 1      allocates BN TMEM columns; one thread issues tcgen05.mma
//               (M=128, N=BN, K=16, bf16 -> fp32 in TMEM) and tcgen05.commit
//               to release each stage and, at the end, the accumulator;
//   warps 2..5  epilogue: tcgen05.ld of their 32 TMEM lanes (= tile rows),
//               round to bf16 (nearest even), 16-byte stores into the row's
//               cache slot (s^K | s^V | z^K | z^V segments).  In the CTAs that
//               hold the positional key's columns they first compute, while the
//               MMAs run, the cosine and sine of every rotated pair of their rows
//               (double precision, on the narrow FP64 pipe), so that after the
//               accumulator lands only the rotation's products remain.
// All waits are bounded (LRKV_DEV_TIMEOUT); no spin is unbounded.
#include "kernels.h"
#include "lrkv_internal.cuh"
#include "rotary.cuh"

namespace lrkv {

namespace {

constexpr int kBM = 128, kBK = 64, kStages = 4;

// Shared memory: the operand ring, the barriers, and (positional key, 128-column tiles) a table
// [pair][2][128 rows] of the rotation's cosines and sines in double -- 64 KB, which fits beside
// the 128 KB ring of 128-column tiles but not the 192 KB one of 256-column tiles; those compute
// the angles in the epilogue instead.
template <int BN, bool ROPE>
struct TcLayout {
    static constexpr uint32_t A_BYTES = kBM * kBK * 2, B_BYTES = BN * kBK * 2;
    static constexpr uint32_t RING = kStages * (A_BYTES + B_BYTES);
    static constexpr bool PRE = ROPE && BN == 128;
    static constexpr uint32_t TAB = RING + 128;
    static constexpr uint32_t SMEM = TAB + (PRE ? 32 * 2 * kBM * 8 : 0) + 1024;
    static_assert(SMEM <= 232448, "fits one CTA's opt-in shared memory");
};

__device__ __forceinline__ long long tc_checked_slot(const AppendArgs& a, int t) {
    const long long s = a.slots[t];
    if (s < 0) return -1;
    if (s >= a.nslots) {
        set_status(a.status, LRKV_DEV_BAD_SLOT);
        return -1;
    }
    return s;
}

// Eight consecutive output columns col..col+7 (never straddling a segment:
// every segment boundary is a multiple of 8) of the row at `slot`.
__device__ __forceinline__ void store8(const AppendArgs& a, long long slot, int col, uint4 v) {
    const int dk = a.d_h + a.d_rope;  // shared key row: [s^K | k^R]
    uint16_t* dst;
    if (col < dk)
        dst = a.sK + slot * dk + col;
    else if (col < dk + a.d_h)
        dst = a.sV + slot * a.d_h + (col - dk);
    else if (col < dk + a.d_h + a.HR)
        dst = a.zK + slot * a.HR + (col - dk - a.d_h);
    else
        dst = a.zV + slot * a.HR + (col - dk - a.d_h - a.HR);
    *reinterpret_cast<uint4*>(dst) = v;
}

}  // namespace

template <int BN, bool ROPE>
__global__ void __launch_bounds__(192, 1)
    append_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const AppendArgs a) {
    constexpr uint32_t A_BYTES = kBM * kBK * 2, B_BYTES = BN * kBK * 2;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + kStages * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * (A_BYTES + B_BYTES));
    uint64_t* empty = full + kStages;
    uint64_t* accf = empty + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kBM;
    const int KT = (a.d + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accf), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % kStages;
                if (kt >= kStages && !mbar_wait(smem_u32(&empty[s]), ((kt / kStages) - 1) & 1, a.status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const uint32_t bar = smem_u32(&full[s]);
                mbar_arrive_expect_tx(bar, A_BYTES + B_BYTES);
                tma_load_2d(sA + s * A_BYTES, &tmX, kt * kBK, m0, bar);
                tma_load_2d(sB + s * B_BYTES, &tmW, kt * kBK, n0, bar);
                issued = kt + 1;
            }
            if (*abort_flag)
                for (int k = max(0, issued - kStages); k < issued; ++k)
                    mbar_wait(smem_u32(&full[k % kStages]), (k / kStages) & 1, a.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % kStages;
                if (*abort_flag || !mbar_wait(smem_u32(&full[s]), (kt / kStages) & 1, a.status)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = sdesc_kmajor_sw128(sA + s * A_BYTES + kk * 32);
                    const uint64_t bd = sdesc_kmajor_sw128(sB + s * B_BYTES + kk * 32);
                    tc_mma_bf16(tmem, ad, bd, idesc, (kt | kk) != 0);
                }
                tc_commit(smem_u32(&empty[s]));
            }
            tc_commit(smem_u32(accf));  // fires once every issued MMA has completed
        }
    } else {
        // epilogue: warps 2..5 -> TMEM lane quarters 2, 3, 0, 1
        const int q = warp & 3;
        constexpr bool PRE = TcLayout<BN, ROPE>::PRE;
        double* tab = reinterpret_cast<double*>(smem + TcLayout<BN, ROPE>::TAB);
        // The positional key's inverse frequencies depend on the pair alone: computed once per
        // CTA (in double, a few dozen operations each on the narrow FP64 pipe) for all rows.
        __shared__ double inv_freq[32];
        const bool rope_cta = ROPE && n0 < a.d_h + a.d_rope && n0 + BN > a.d_h;
        const int i0 = rope_cta ? (max(n0, a.d_h) - a.d_h) / 2 : 0;  // first pair of this CTA
        if (rope_cta) {
            const int t = threadIdx.x - 64;
            if (t < a.d_rope / 2 && t < 32) inv_freq[t] = rope_inv_freq(t, a.d_rope, a.rope_base);
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
            if (PRE) {
                // cosine and sine of each rotated pair of this thread's row, while the MMAs run
                const int row = m0 + q * 32 + lane;
                const int i1 = (min(n0 + BN, a.d_h + a.d_rope) - a.d_h) / 2;
                if (row < a.n) {
                    const int pos = a.positions[row];
                    for (int i = i0; i < i1; ++i) {
                        double cs, sn;
                        rope_cos_sin(inv_freq[i], pos, cs, sn);
                        tab[(2 * (i - i0)) * kBM + q * 32 + lane] = cs;
                        tab[(2 * (i - i0) + 1) * kBM + q * 32 + lane] = sn;
                    }
                }
            }
        }
        bool ok = mbar_wait(smem_u32(accf), 0, a.status);
        ok = __all_sync(0xffffffffu, ok && !*abort_flag);  // warp-uniform: tcgen05.ld below is warp-collective
        tc_fence_after();
        if (ok) {
            const int row = m0 + q * 32 + lane;
            const long long slot = row < a.n ? tc_checked_slot(a, row) : -1;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
                // Columns of the shared positional key (a 32-aligned range [d_h, d_h + d_rope))
                // are rotated at the row's position before rounding.
                if (ROPE && slot >= 0 && n0 + c0 >= a.d_h && n0 + c0 < a.d_h + a.d_rope) {
                    const int pos = a.positions[row];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0 = __uint_as_float(v[2 * e]), x1 = __uint_as_float(v[2 * e + 1]);
                        const int i = (n0 + c0 - a.d_h) / 2 + e;
                        if (PRE)
                            rope_apply(x0, x1, tab[(2 * (i - i0)) * kBM + q * 32 + lane],
                                       tab[(2 * (i - i0) + 1) * kBM + q * 32 + lane]);
                        else
                            rope_rotate_f(x0, x1, inv_freq[i], pos);
                        v[2 * e] = __float_as_uint(x0);
                        v[2 * e + 1] = __float_as_uint(x1);
                    }
                }
                if (slot >= 0) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = n0 + c0 + g * 8;
                        if (col < a.N) {
                            uint4 pk;
                            pk.x = pack_bf16x2(__uint_as_float(v[g * 8 + 0]), __uint_as_float(v[g * 8 + 1]));
                            pk.y = pack_bf16x2(__uint_as_float(v[g * 8 + 2]), __uint_as_float(v[g * 8 + 3]));
                            pk.z = pack_bf16x2(__uint_as_float(v[g * 8 + 4]), __uint_as_float(v[g * 8 + 5]));
                            pk.w = pack_bf16x2(__uint_as_float(v[g * 8 + 6]), __uint_as_float(v[g * 8 + 7]));
                            store8(a, slot, col, pk);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, BN);
    }
}

template <int BN, bool ROPE>
static cudaError_t launch_tc(const CUtensorMap& tmX, const CUtensorMap& tmW, const AppendArgs& a,
                             cudaStream_t stream) {
    constexpr int smem = TcLayout<BN, ROPE>::SMEM;
    auto kern = append_tc_kernel<BN, ROPE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + BN - 1) / BN, (a.n + kBM - 1) / kBM);
    kern<<<grid, 192, smem, stream>>>(tmX, tmW, a);
    return cudaGetLastError();
}

int append_tc_block_n(int N) { return (N % 256 == 0) ? 256 : 128; }

cudaError_t launch_append_tc(const CUtensorMap& tmX, const CUtensorMap& tmW, const AppendArgs& a,
                             cudaStream_t stream) {
    // the positional-key rotation is compiled only into the kernels that need it
    if (a.d_rope > 0)
        return append_tc_block_n(a.N) == 256 ? launch_tc<256, true>(tmX, tmW, a, stream)
                                             : launch_tc<128, true>(tmX, tmW, a, stream);
    return append_tc_block_n(a.N) == 256 ? launch_tc<256, false>(tmX, tmW, a, stream)
                                         : launch_tc<128, false>(tmX, tmW, a, stream);
}

}  // namespace lrkv
