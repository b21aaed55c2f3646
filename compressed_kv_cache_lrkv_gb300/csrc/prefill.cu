// prefill.cu -- causal chunked prefill over the LRKV cache ("Low-Rank Key Value
// Attention", Eqs. (6)-(7) with the causal mask of the softmax frame).
//
// For head h the logits of query i against key j are the dot product of the
// concatenated rows [q_i | q~_i] . [s^K_j | z^K_{h,j}] (width d_h + r), with
// q~_i = q_i B_h^K; the value side accumulates P [s^V | z^V_h] into (o_s, o_z)
// and the epilogue returns o_s + B_h^V o_z.  With absorbed weights (a.qt set) q~
// comes from the caller and the epilogue returns [o_s | o_z] instead.  Query i sits at absolute position
// q_start + i and sees keys j <= q_start + i.  With a decoupled positional key
// (D_R > 0) the shared key row is [s^K | k^R] and the query [q | q^R]: the
// shared logits run over D_K = D_H + D_R columns, q~ uses the first D_H.
//
// One CTA = 64 queries of one (sequence, head); four warps of 16 query rows
// each run a flash-attention loop over 64-token key tiles (one cache page per
// tile), double-buffered with cp.async, on warp-level tensor-core MMAs
// (m16n8k16 bf16, fp32 accumulate).  Rows beyond the context are zero-filled
// so masked tokens can never inject NaN through 0 * garbage.
#include "kernels.h"
#include "lrkv_internal.cuh"

namespace lrkv {

namespace {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Row pitch (bytes) of a padded shared-memory tile: an odd number of 16-byte
// chunks, so eight ldmatrix rows land in eight distinct bank groups.
constexpr int padded_pitch(int row_bytes) { return ((row_bytes / 16) % 2 == 1) ? row_bytes : row_bytes + 16; }

}  // namespace

template <int D_H, int R, int D_R>
struct PrefillTile {
    static constexpr int kTok = 64;
    static constexpr int kPitchK = padded_pitch((D_H + D_R) * 2);  // key rows [s^K | k^R]
    static constexpr int kPitchS = padded_pitch(D_H * 2);          // value rows s^V
    static constexpr int kPitchZ = padded_pitch(R * 2);
    static constexpr int kKBytes = kTok * kPitchK;
    static constexpr int kSBytes = kTok * kPitchS;
    static constexpr int kZBytes = kTok * kPitchZ;
    static constexpr int kStage = kKBytes + kSBytes + 2 * kZBytes;
    static constexpr int kScratch = 4 * 16 * R * 4;  // per-warp [16][R] fp32
    static constexpr int kSmem = 2 * kStage + kScratch;
};

template <int D_H, int R, int D_R>
__global__ void __launch_bounds__(128) prefill_kernel(const PrefillArgs a) {
    using T = PrefillTile<D_H, R, D_R>;
    constexpr int D_K = D_H + D_R;
    extern __shared__ __align__(16) uint8_t smem[];
    const uint32_t smem_s = smem_u32(smem);
    const int qtile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int H = a.H, Tq = a.Tq;
    const int qs = a.q_start[b];
    const int ctx = qs + Tq;
    const int cap = a.max_pages * kBlockSize;
    const int i0 = qtile * 64 + warp * 16;  // this warp's first query row
    const int rA = i0 + g, rB = i0 + g + 8;

    const bool fused = a.qt != nullptr;
    const int ow = fused ? D_H + R : D_H;  // output row width
    auto out_row = [&](int i) { return a.out + (((size_t)b * Tq + i) * H + h) * ow; };
    if (qs < 0 || ctx > cap) {
        if (threadIdx.x == 0 && qtile == 0 && h == 0) set_status(a.status, LRKV_DEV_BAD_SEQLEN);
        for (int idx = threadIdx.x; idx < 64 * ow; idx += 128) {
            const int i = qtile * 64 + idx / ow;
            if (i < Tq) out_row(i)[idx % ow] = 0;
        }
        return;
    }
    const int last_row = min(qtile * 64 + 63, Tq - 1);
    const int n_tiles = (qs + last_row) / 64 + 1;

    // ---- q fragments and q~ = q B_h^K (fp32, rounded to bf16 for the MMA), or the caller's q~
    uint32_t qa[D_K / 16][4];
    {
        const uint32_t* qA = reinterpret_cast<const uint32_t*>(a.q + (((size_t)b * Tq + rA) * H + h) * D_K);
        const uint32_t* qB = reinterpret_cast<const uint32_t*>(a.q + (((size_t)b * Tq + rB) * H + h) * D_K);
#pragma unroll
        for (int kk = 0; kk < D_K / 16; ++kk) {
            qa[kk][0] = rA < Tq ? qA[kk * 8 + tq] : 0u;
            qa[kk][1] = rB < Tq ? qB[kk * 8 + tq] : 0u;
            qa[kk][2] = rA < Tq ? qA[kk * 8 + 4 + tq] : 0u;
            qa[kk][3] = rB < Tq ? qB[kk * 8 + 4 + tq] : 0u;
        }
    }
    float* wscr = reinterpret_cast<float*>(smem + 2 * T::kStage) + warp * 16 * R;
    {
        const int row = lane & 15, jh = lane >> 4;
        const int i = i0 + row;
        const size_t qi = ((size_t)b * Tq + min(i, Tq - 1)) * H + h;
        const uint16_t* qrow = a.q + qi * D_K;
        for (int j = jh * (R / 2); j < (jh + 1) * (R / 2); ++j) {
            float acc = 0.f;
            if (fused) {
                acc = __uint_as_float((uint32_t)a.qt[qi * R + j] << 16);
            } else {
                const uint16_t* bk = a.BK + (size_t)h * D_H * R + j;
                for (int dd = 0; dd < D_H; ++dd)
                    acc = fmaf(__uint_as_float((uint32_t)qrow[dd] << 16), __uint_as_float((uint32_t)bk[dd * R] << 16),
                               acc);
            }
            wscr[row * R + j] = i < Tq ? acc : 0.f;
        }
    }
    __syncwarp();
    constexpr int KZ = (R + 15) / 16;  // k16 steps of the residual logits (R = 8 uses one m16n8k8)
    uint32_t qza[KZ][4];
#pragma unroll
    for (int kz = 0; kz < KZ; ++kz) {
        const int c0 = kz * 16 + 2 * tq;
        qza[kz][0] = pack_bf16x2(wscr[g * R + c0], wscr[g * R + c0 + 1]);
        qza[kz][1] = pack_bf16x2(wscr[(g + 8) * R + c0], wscr[(g + 8) * R + c0 + 1]);
        if (R >= 16) {
            qza[kz][2] = pack_bf16x2(wscr[g * R + c0 + 8], wscr[g * R + c0 + 9]);
            qza[kz][3] = pack_bf16x2(wscr[(g + 8) * R + c0 + 8], wscr[(g + 8) * R + c0 + 9]);
        } else {
            qza[kz][2] = qza[kz][3] = 0u;
        }
    }

    // ---- tile loader: 64 tokens of [s^K | k^R], s^V and z^K_h, z^V_h (r) for head h
    auto load_tile = [&](int kt, int buf) {
        const uint32_t st = smem_s + buf * T::kStage;
        int blk = a.block_table[(size_t)b * a.max_pages + kt];
        bool ok = true;
        if (blk < 0 || blk >= a.num_blocks) {
            ok = false;
            if (threadIdx.x == 0) set_status(a.status, LRKV_DEV_BAD_BLOCK);
            blk = 0;
        }
        constexpr int CK = D_K / 8, CS = D_H / 8, CZ = R / 8;
        if (D_R > 0) {
            for (int idx = threadIdx.x; idx < 64 * CK; idx += 128) {
                const int tok = idx / CK, c = idx % CK;
                const bool live = ok && (kt * 64 + tok < ctx);
                cp_async16(st + tok * T::kPitchK + c * 16, a.sK + ((size_t)blk * 64 + tok) * D_K + c * 8, live ? 16 : 0);
            }
        }
        for (int idx = threadIdx.x; idx < 64 * CS; idx += 128) {
            const int tok = idx / CS, c = idx % CS;
            const bool live = ok && (kt * 64 + tok < ctx);
            const size_t go = ((size_t)blk * 64 + tok) * D_H + c * 8;
            if (D_R == 0) cp_async16(st + tok * T::kPitchK + c * 16, a.sK + go, live ? 16 : 0);
            cp_async16(st + T::kKBytes + tok * T::kPitchS + c * 16, a.sV + go, live ? 16 : 0);
        }
        for (int idx = threadIdx.x; idx < 64 * CZ; idx += 128) {
            const int tok = idx / CZ, c = idx % CZ;
            const bool live = ok && (kt * 64 + tok < ctx);
            const size_t go = (((size_t)blk * 64 + tok) * H + h) * R + c * 8;
            cp_async16(st + T::kKBytes + T::kSBytes + tok * T::kPitchZ + c * 16, a.zK + go, live ? 16 : 0);
            cp_async16(st + T::kKBytes + T::kSBytes + T::kZBytes + tok * T::kPitchZ + c * 16, a.zV + go,
                       live ? 16 : 0);
        }
    };

    float os[D_H / 8][4];
    float oz[R / 8][4];
#pragma unroll
    for (int n = 0; n < D_H / 8; ++n) os[n][0] = os[n][1] = os[n][2] = os[n][3] = 0.f;
#pragma unroll
    for (int n = 0; n < R / 8; ++n) oz[n][0] = oz[n][1] = oz[n][2] = oz[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int posA = qs + min(rA, Tq - 1), posB = qs + min(rB, Tq - 1);
    const int warp_last_pos = qs + min(i0 + 15, Tq - 1);

    load_tile(0, 0);
    cp_async_commit();
    for (int kt = 0; kt < n_tiles; ++kt) {
        if (kt + 1 < n_tiles) load_tile(kt + 1, (kt + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int buf = kt & 1;
        const uint32_t sK_s = smem_s + buf * T::kStage;
        const uint32_t sV_s = sK_s + T::kKBytes;
        const uint32_t zK_s = sV_s + T::kSBytes;
        const uint32_t zV_s = zK_s + T::kZBytes;
        const int key0 = kt * 64;
        if (i0 < Tq && key0 <= warp_last_pos) {
            // ---- logits S[16 x 64]
            float s[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
                const int tok = nt * 8 + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < D_K / 16; kk += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(sK_s + tok * T::kPitchK + (kk * 2 + (lane >> 3)) * 16, b0, b1, b2, b3);
                    mma_16816(s[nt], qa[kk], b0, b1);
                    mma_16816(s[nt], qa[kk + 1], b2, b3);
                }
                if (R >= 16) {
#pragma unroll
                    for (int kz = 0; kz < KZ; ++kz) {
                        uint32_t b0, b1, b2, b3;
                        // matrices: chunks 2kz, 2kz+1 of these 8 tokens (x4 reads them twice; use the first two)
                        ldmatrix_x4(zK_s + tok * T::kPitchZ + ((kz * 2 + ((lane >> 3) & 1)) * 16), b0, b1, b2, b3);
                        mma_16816(s[nt], qza[kz], b0, b1);
                    }
                } else {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(zK_s + tok * T::kPitchZ, b0, b1, b2, b3);
                    mma_1688(s[nt], qza[0][0], qza[0][1], b0);
                }
            }
            // ---- causal mask, online softmax (log2 domain)
            const bool diag = key0 + 63 > qs + i0;
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int j = key0 + nt * 8 + 2 * tq;
                s[nt][0] = (!diag || j <= posA) ? s[nt][0] * a.scale_log2 : -INFINITY;
                s[nt][1] = (!diag || j + 1 <= posA) ? s[nt][1] * a.scale_log2 : -INFINITY;
                s[nt][2] = (!diag || j <= posB) ? s[nt][2] * a.scale_log2 : -INFINITY;
                s[nt][3] = (!diag || j + 1 <= posB) ? s[nt][3] * a.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
            const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                s[nt][0] = (mn0 == -INFINITY) ? 0.f : exp2f(s[nt][0] - mn0);
                s[nt][1] = (mn0 == -INFINITY) ? 0.f : exp2f(s[nt][1] - mn0);
                s[nt][2] = (mn1 == -INFINITY) ? 0.f : exp2f(s[nt][2] - mn1);
                s[nt][3] = (mn1 == -INFINITY) ? 0.f : exp2f(s[nt][3] - mn1);
                rs0 += s[nt][0] + s[nt][1];
                rs1 += s[nt][2] + s[nt][3];
            }
            m0 = mn0;
            m1 = mn1;
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
#pragma unroll
            for (int n = 0; n < D_H / 8; ++n) {
                os[n][0] *= al0; os[n][1] *= al0; os[n][2] *= al1; os[n][3] *= al1;
            }
#pragma unroll
            for (int n = 0; n < R / 8; ++n) {
                oz[n][0] *= al0; oz[n][1] *= al0; oz[n][2] *= al1; oz[n][3] *= al1;
            }
            // ---- P [s^V | z^V_h]
#pragma unroll
            for (int kc = 0; kc < 4; ++kc) {
                uint32_t pa[4];
                pa[0] = pack_bf16x2(s[2 * kc][0], s[2 * kc][1]);
                pa[1] = pack_bf16x2(s[2 * kc][2], s[2 * kc][3]);
                pa[2] = pack_bf16x2(s[2 * kc + 1][0], s[2 * kc + 1][1]);
                pa[3] = pack_bf16x2(s[2 * kc + 1][2], s[2 * kc + 1][3]);
                const int mi = lane >> 3;
                const int tok = kc * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int dn = 0; dn < D_H / 8; dn += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(sV_s + tok * T::kPitchS + (dn + (mi >> 1)) * 16, b0, b1, b2, b3);
                    mma_16816(os[dn], pa, b0, b1);
                    mma_16816(os[dn + 1], pa, b2, b3);
                }
#pragma unroll
                for (int zn = 0; zn < R / 8; zn += 2) {
                    uint32_t b0, b1, b2, b3;
                    const int chunk = (R >= 16) ? zn + (mi >> 1) : 0;
                    ldmatrix_x4_trans(zV_s + tok * T::kPitchZ + chunk * 16, b0, b1, b2, b3);
                    mma_16816(oz[zn], pa, b0, b1);
                    if (zn + 1 < R / 8) mma_16816(oz[zn + 1], pa, b2, b3);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- epilogue: out = (o_s + B_h^V o_z) / l
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    if (fused) {  // [o_s | o_z] / l
#pragma unroll
        for (int n = 0; n < D_H / 8; ++n) {
            const int dcol = n * 8 + 2 * tq;
            if (rA < Tq) *reinterpret_cast<uint32_t*>(out_row(rA) + dcol) = pack_bf16x2(os[n][0] * inv0, os[n][1] * inv0);
            if (rB < Tq) *reinterpret_cast<uint32_t*>(out_row(rB) + dcol) = pack_bf16x2(os[n][2] * inv1, os[n][3] * inv1);
        }
#pragma unroll
        for (int n = 0; n < R / 8; ++n) {
            const int zcol = D_H + n * 8 + 2 * tq;
            if (rA < Tq) *reinterpret_cast<uint32_t*>(out_row(rA) + zcol) = pack_bf16x2(oz[n][0] * inv0, oz[n][1] * inv0);
            if (rB < Tq) *reinterpret_cast<uint32_t*>(out_row(rB) + zcol) = pack_bf16x2(oz[n][2] * inv1, oz[n][3] * inv1);
        }
        return;
    }
    __syncwarp();
#pragma unroll
    for (int n = 0; n < R / 8; ++n) {
        wscr[g * R + n * 8 + 2 * tq] = oz[n][0];
        wscr[g * R + n * 8 + 2 * tq + 1] = oz[n][1];
        wscr[(g + 8) * R + n * 8 + 2 * tq] = oz[n][2];
        wscr[(g + 8) * R + n * 8 + 2 * tq + 1] = oz[n][3];
    }
    __syncwarp();
    const uint16_t* bv = a.BV + (size_t)h * D_H * R;
#pragma unroll
    for (int n = 0; n < D_H / 8; ++n) {
        const int dcol = n * 8 + 2 * tq;
        float v[4] = {os[n][0], os[n][1], os[n][2], os[n][3]};
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float b0 = __uint_as_float((uint32_t)bv[(size_t)dcol * R + j] << 16);
            const float b1 = __uint_as_float((uint32_t)bv[(size_t)(dcol + 1) * R + j] << 16);
            v[0] = fmaf(b0, wscr[g * R + j], v[0]);
            v[1] = fmaf(b1, wscr[g * R + j], v[1]);
            v[2] = fmaf(b0, wscr[(g + 8) * R + j], v[2]);
            v[3] = fmaf(b1, wscr[(g + 8) * R + j], v[3]);
        }
        if (rA < Tq) *reinterpret_cast<uint32_t*>(out_row(rA) + dcol) = pack_bf16x2(v[0] * inv0, v[1] * inv0);
        if (rB < Tq) *reinterpret_cast<uint32_t*>(out_row(rB) + dcol) = pack_bf16x2(v[2] * inv1, v[3] * inv1);
    }
}

template <int D_H, int R, int D_R>
static cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
    using T = PrefillTile<D_H, R, D_R>;
    auto kern = prefill_kernel<D_H, R, D_R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.Tq + 63) / 64, a.H, a.B);
    kern<<<grid, 128, T::kSmem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, int D_H, int R, int D_R, cudaStream_t stream) {
#define LRKV_PF(DH, RR)                                                                                  \
    if (D_H == DH && R == RR)                                                                            \
        return D_R == 0 ? launch_prefill_t<DH, RR, 0>(a, stream) : launch_prefill_t<DH, RR, 64>(a, stream);
    LRKV_PF(64, 8) LRKV_PF(64, 16) LRKV_PF(64, 32) LRKV_PF(128, 8) LRKV_PF(128, 16) LRKV_PF(128, 32)
#undef LRKV_PF
    return cudaErrorInvalidValue;
}

}  // namespace lrkv
