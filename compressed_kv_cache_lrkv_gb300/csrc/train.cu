// train.cu -- training-time forward and backward of one expanded LRKV projection
// ("Low-Rank Key Value Attention", frame "Training learns the base and residuals together":
// the full per-head features are materialised, K_h = X W_h with W_h = W_shared + U_h B_h^T,
// Eqs. (2)-(3)).  Keys and values are the same operation with their own factors.
//
// Forward (W_T = [W_shared^T ; U_1^T ; ... ; U_H^T], [d_h + H r][d]):
//   Y = X W_T^T = [S | R_1 .. R_H]            one GEMM, N = d_h + H r
//   K_h = S + R_h B_h^T = [S | R_h] [I ; B_h^T]  per head, K = d_h + r: the shared part enters the
//                                                product through an identity block, so S and R_h B_h^T
//                                                are summed in fp32 and rounded once (B_h's box past r
//                                                reads zeros)
// Backward, for dK [n][H][d_h]:
//   Gc = [G | dR_1 .. dR_H], G = sum_h dK_h, dR_h = dK_h B_h
//   dB_h = dK_h^T R_h                            per 128-token tile, fp32 partials, ordered sum
//   dW_T = Gc^T X                                (= [dW_shared^T ; dU_1^T ; ...]), K = n
//   dX = Gc W_T                                  K = d_h + H r
// All contractions run on tcgen05 (bf16 operands, fp32 accumulation in TMEM); S, R and Gc are
// rounded to bf16 between the steps, as the inference cache rounds S and R.
//
// tgemm_kernel: a persistent GEMM (one CTA per SM looping over 128 x BN output tiles of up to two
// products, round robin or from a shared work queue): warp 0 TMA producer (a ring of 64-wide K
// slices, continuous across tiles), warp 1 TMEM owner and single-thread MMA issue into one of two
// accumulator buffers, warps 2-5 epilogue (tcgen05.ld of their 32 TMEM lanes = tile rows), so a
// tile's epilogue overlaps the next tile's MMAs.  A bf16 tile leaves through shared memory: each
// epilogue warp writes its 32 rows into 32 x 32 boxes (64-byte swizzle, conflict-free 16-byte
// stores) and one lane issues their TMA stores.
// dk_pass_kernel: the backward's one pass over dK on CTA pairs (G in registers, dR and the dB
// partials on the tensor cores), described at the kernel.  All waits are bounded.
#include "kernels.h"
#include "lrkv_internal.cuh"
#include "train.h"

#include <cstring>

namespace lrkv {

namespace {

constexpr int kTM = 128, kTK = 64;
constexpr uint32_t T_A = kTM * kTK * 2;  // 16 KiB: 128 rows x 64 K
constexpr uint32_t kTBox = 2048;         // staging box: 32 rows x 32 bf16 columns (64 bytes)
constexpr uint32_t kTSmemMax = 232448;   // opt-in shared memory per block

// Per output-tile width BN: bytes of one B slice, staging boxes per epilogue warp, ring depth,
// TMEM columns.
template <int BN>
struct TCfg {
    static constexpr uint32_t B = (uint32_t)BN * kTK * 2;
    static constexpr int NBOX = 4;
    static constexpr uint32_t STG = 4u * NBOX * kTBox;
    static constexpr int S0 = (int)((kTSmemMax - 1280 - STG) / (T_A + B));
    static constexpr int STAGES = S0 > 8 ? 8 : S0;
    static constexpr uint32_t SMEM = STAGES * (T_A + B) + STG + 256 + 1024;
    static constexpr uint32_t TMEM = 2 * BN <= 256 ? 256 : 512;
};

// K-major operand: rows x 64 K, 128-byte swizzle, 8-row groups 1 KiB apart.  MN-major operand:
// 64-wide blocks of [64 K rows][128 B], 8 KiB apart, 8-row K groups 1 KiB apart.
__device__ __forceinline__ uint64_t kmaj(uint32_t a) { return sdesc(a, 16, 1024, 2); }
__device__ __forceinline__ uint64_t mnmaj(uint32_t a) { return sdesc(a, 8192, 1024, 2); }

// Tiled store shared -> global (bulk-group completion); the box is clipped at the tensor's extents.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's committed bulk stores still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until this thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// A 128 x 128 bf16 identity, the B block that adds the shared features S into the expansion.
struct IdentityBf16 {
    uint16_t v[128 * 128];
    constexpr IdentityBf16() : v() {
        for (int i = 0; i < 128; ++i) v[i * 129] = 0x3F80;  // 1.0
    }
};
__device__ const IdentityBf16 g_identity{};

}  // namespace

const void* train_identity() {
    void* p = nullptr;
    return cudaGetSymbolAddress(&p, g_identity) == cudaSuccess ? p : nullptr;
}

template <bool OUTF32, int BN, bool GROUPED>
__global__ void __launch_bounds__(192, 1) tgemm_kernel(const __grid_constant__ TGemmParams p) {
    using C = TCfg<BN>;
    constexpr int kS = C::STAGES, NBOX = C::NBOX;
    constexpr uint32_t T_B = C::B;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + kS * T_A;
    uint8_t* stg_base = smem + kS * (T_A + T_B);  // epilogue staging, 1 KiB aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(stg_base + C::STG);
    uint64_t* empty = full + kS;
    uint64_t* acc_full = empty + kS;      // [2] accumulator buffer holds a finished tile
    uint64_t* acc_empty = acc_full + 2;   // [2] the epilogue has read it (128 arrivals)
    uint64_t* wq_full = acc_empty + 2;    // [4] work queue: the producer published an item
    uint64_t* wq_empty = wq_full + 4;     // [4] the MMA thread and the 4 epilogue warps read it
    int* wq = reinterpret_cast<int*>(wq_empty + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wq + 4);
    volatile int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    uint32_t* status = p.g[0].status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool dyn = GROUPED && p.ctr != nullptr;
    // work item -> (group, n tile, m tile, batch, k split); n fastest, so consecutive items share
    // A rows in L2; group 0's items come first
    struct Tile {
        int grp, n0, m0, z, batch, kt0, KT;
    };
    auto tile_of = [&](int w) {
        Tile r;
        r.grp = GROUPED && w >= p.tiles0 ? 1 : 0;
        const GemmArgs& g = p.g[r.grp];
        const int t = w - (r.grp ? p.tiles0 : 0);
        const int tiles_n = (g.N + BN - 1) / BN, tiles_m = (g.M + kTM - 1) / kTM;
        const int KT_all = (g.K + kTK - 1) / kTK;
        const int per = (KT_all + g.ksplit - 1) / g.ksplit;
        r.n0 = (t % tiles_n) * BN;
        r.m0 = ((t / tiles_n) % tiles_m) * kTM;
        r.z = t / (tiles_n * tiles_m);
        r.batch = r.z / g.ksplit;
        r.kt0 = (r.z % g.ksplit) * per;
        r.KT = max(0, min(KT_all, r.kt0 + per) - r.kt0);
        return r;
    };
    // Work item of local iteration `it` for the MMA thread and the epilogue: the round-robin one,
    // or the one the producer took from the queue (returns total at the end; arrives as reader)
    auto next_item = [&](int it, bool lead, bool& ok) -> int {
        if (!dyn) return blockIdx.x + it * gridDim.x < p.total ? (int)(blockIdx.x + it * gridDim.x) : p.total;
        ok = ok && mbar_wait(smem_u32(&wq_full[it & 3]), (it >> 2) & 1, status);
        const int w = ok ? wq[it & 3] : p.total;
        if (lead) mbar_arrive(smem_u32(&wq_empty[it & 3]));
        return w;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 128);
        }
        for (int q = 0; q < 4; ++q) {
            mbar_init(smem_u32(&wq_full[q]), 1);
            mbar_init(smem_u32(&wq_empty[q]), 5);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int q = 0;  // K slices issued by this CTA (ring position and phase)
            bool ok = true;
            for (int it = 0; ok; ++it) {
                int w;
                if (dyn) {
                    // take the next item and publish it (the first one is this CTA's own)
                    w = it == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.ctr, 1);
                    if (w > p.total) w = p.total;
                    if (it >= 4 && !mbar_wait(smem_u32(&wq_empty[it & 3]), ((it >> 2) - 1) & 1, status)) {
                        *abort_flag = 1;
                        break;
                    }
                    wq[it & 3] = w;
                    mbar_arrive(smem_u32(&wq_full[it & 3]));
                } else {
                    w = blockIdx.x + it * gridDim.x;
                }
                if (w >= p.total) break;
                const Tile tl = tile_of(w);
                const GemmArgs& g = p.g[tl.grp];
                const CUtensorMap* mA = GROUPED && tl.grp ? &p.A[1] : &p.A[0];
                const CUtensorMap* mB = GROUPED && tl.grp ? &p.B[1] : &p.B[0];
                const int ax = g.a_x0 + tl.batch * g.a_zx, ay = g.a_y0 + tl.batch * g.a_zy;
                const int bx = g.b_x0 + tl.batch * g.b_zx, by = g.b_y0 + tl.batch * g.b_zy;
                const bool amn = g.a_mn != 0, bmn = g.b_mn != 0;
                const int kfix = (amn || bmn) ? 0 : g.kfix;
                for (int i = 0; i < tl.KT; ++i, ++q) {
                    const int s = q % kS;
                    if ((q >= kS && !mbar_wait(smem_u32(&empty[s]), ((q / kS) - 1) & 1, status)) || *abort_flag) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    const int k = (tl.kt0 + i) * kTK;
                    const uint32_t bar = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(bar, T_A + T_B);
                    if (k < kfix) {
                        // leading K columns shared by every batch: A at x = k, B from the second map
                        tma_load_2d(sA + s * T_A, mA, k, ay + tl.m0, bar);
                        tma_load_2d(sB + s * T_B, &p.B2, k, tl.n0, bar);
                        continue;
                    }
                    const int kb = k - kfix;
                    if (amn) {
                        tma_load_2d(sA + s * T_A, mA, ax + tl.m0, ay + k, bar);
                        tma_load_2d(sA + s * T_A + 8192, mA, ax + tl.m0 + 64, ay + k, bar);
                    } else {
                        tma_load_2d(sA + s * T_A, mA, ax + kb, ay + tl.m0, bar);
                    }
                    if (bmn) {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j) tma_load_2d(sB + s * T_B + j * 8192, mB, bx + tl.n0 + 64 * j, by + k, bar);
                    } else {
                        tma_load_2d(sB + s * T_B, mB, bx + kb, by + tl.n0, bar);  // one [BN][64] box
                    }
                }
            }
            if (*abort_flag)  // let the copies in flight land before the CTA exits
                for (int k = max(0, q - kS); k < q; ++k) mbar_wait(smem_u32(&full[k % kS]), (k / kS) & 1, status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc0 = idesc_bf16_f32(kTM, BN);
            int q = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int w = next_item(it, true, ok);
                if (!ok || w >= p.total) break;
                const Tile tl = tile_of(w);
                const bool amn = p.g[tl.grp].a_mn != 0, bmn = p.g[tl.grp].b_mn != 0;
                const uint32_t idesc = idesc0 | ((uint32_t)amn << 15) | ((uint32_t)bmn << 16);
                // descriptor of K step 0 and the per-step advance (16 B in the encoded start address
                // field per 16 elements: 2 for a K-major row step of 32 B, 128 for 2 KiB of an MN-major block)
                const uint64_t a_base = amn ? mnmaj(sA) : kmaj(sA), b_base = bmn ? mnmaj(sB) : kmaj(sB);
                const uint64_t a_kk = amn ? 128 : 2, b_kk = bmn ? 128 : 2;
                const int buf = it & 1;
                // the epilogue must have read this buffer's previous tile
                if (it >= 2 && !mbar_wait(smem_u32(&acc_empty[buf]), ((it >> 1) - 1) & 1, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + buf * BN;
                for (int i = 0; i < tl.KT; ++i, ++q) {
                    const int s = q % kS;
                    if (*abort_flag || !mbar_wait(smem_u32(&full[s]), (q / kS) & 1, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_s = a_base + (uint64_t)((s * T_A) >> 4), b_s = b_base + (uint64_t)((s * T_B) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTK / 16; ++kk)
                        tc_mma_bf16(acc, a_s + kk * a_kk, b_s + kk * b_kk, idesc, (i | kk) != 0);
                    tc_commit(smem_u32(&empty[s]));
                }
                if (!ok) break;
                tc_commit(smem_u32(&acc_full[buf]));  // fires once this tile's MMAs have completed
            }
            if (!ok) *abort_flag = 1;
        }
    } else {
        // epilogue: warps 2..5 -> TMEM lane quarters 2, 3, 0, 1.  Each warp stages its 32 rows of a
        // 32-column chunk in a 2 KiB box (64-byte swizzle: 16-byte chunk j of row i sits at
        // j ^ ((i >> 1) & 3), so the 16-byte stores are conflict-free) and one lane stores the box
        // by TMA; the boxes form a ring per warp.
        const int q4 = warp & 3;
        uint8_t* stg = stg_base + q4 * (NBOX * kTBox);
        const uint32_t stg_s = smem_u32(stg);
        const int swz = (lane >> 1) & 3;
        int qc = 0;
        bool used_tma = false;
        bool okq = true;
        for (int it = 0;; ++it) {
            int w = next_item(it, false, okq);
            __syncwarp();
            if (dyn && lane == 0) mbar_arrive(smem_u32(&wq_empty[it & 3]));
            if (!okq || w >= p.total) break;
            const Tile tl = tile_of(w);
            const GemmArgs& g = p.g[tl.grp];
            const bool tma = !OUTF32 && g.tma_out;
            const CUtensorMap* mC = GROUPED && tl.grp ? &p.C[1] : &p.C[0];
            const int buf = it & 1;
            const int ry = tl.m0 + q4 * 32;  // this warp's first output row
            bool ok = !*abort_flag && mbar_wait(smem_u32(&acc_full[buf]), (it >> 1) & 1, status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int row = ry + lane;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32, ++qc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + buf * BN + ((uint32_t)(q4 * 32) << 16) + c0, v);
                if (tl.KT == 0)
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                if (tma) {
                    used_tma = true;
                    const int box = qc % NBOX;
                    if (lane == 0) bulk_wait_read<NBOX - 1>();  // the store that last used this box has read it
                    __syncwarp();
                    uint8_t* rowp = stg + box * kTBox + lane * 64;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 pk;
                        pk.x = pack_bf16x2(__uint_as_float(v[j * 8 + 0]), __uint_as_float(v[j * 8 + 1]));
                        pk.y = pack_bf16x2(__uint_as_float(v[j * 8 + 2]), __uint_as_float(v[j * 8 + 3]));
                        pk.z = pack_bf16x2(__uint_as_float(v[j * 8 + 4]), __uint_as_float(v[j * 8 + 5]));
                        pk.w = pack_bf16x2(__uint_as_float(v[j * 8 + 6]), __uint_as_float(v[j * 8 + 7]));
                        *reinterpret_cast<uint4*>(rowp + ((j ^ swz) << 4)) = pk;
                    }
                    fence_proxy_async_smem();  // the generic stores above, before the async-proxy read
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(mC, stg_s + box * kTBox, tl.n0 + c0, tl.batch, ry);
                        bulk_commit();
                    }
                } else if (OUTF32) {
                    // split-K partial of a single-tile product: [batch][ks][128][BN] fp32
                    float* dst = reinterpret_cast<float*>(g.C) + (((size_t)tl.z * kTM + (row - tl.m0)) * BN + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        reinterpret_cast<float4*>(dst)[i] =
                            make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                        __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                } else if (row < g.M) {
                    uint16_t* crow = reinterpret_cast<uint16_t*>(g.C) + tl.batch * g.c_zstride + (size_t)row * g.ldc;
#pragma unroll
                    for (int gi = 0; gi < 4; ++gi) {
                        const int col = tl.n0 + c0 + gi * 8;
                        if (col < g.N) {
                            uint4 pk;
                            pk.x = pack_bf16x2(__uint_as_float(v[gi * 8 + 0]), __uint_as_float(v[gi * 8 + 1]));
                            pk.y = pack_bf16x2(__uint_as_float(v[gi * 8 + 2]), __uint_as_float(v[gi * 8 + 3]));
                            pk.z = pack_bf16x2(__uint_as_float(v[gi * 8 + 4]), __uint_as_float(v[gi * 8 + 5]));
                            pk.w = pack_bf16x2(__uint_as_float(v[gi * 8 + 6]), __uint_as_float(v[gi * 8 + 7]));
                            *reinterpret_cast<uint4*>(crow + col) = pk;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&acc_empty[buf]));
        }
        if (used_tma && lane == 0) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM);
    }
}

// ------------------------------------------------------------------ fused pass over dK
// For one 128-token tile: G = sum_h dK_h (Gc columns [0, d_h)) and dR_h = dK_h B_h (Gc columns
// d_h + h r ..), and with dB folded in (d_h = 128, r = 16) this tile's part of every
// dB_h = dK_h^T R_h, reading each dK_h tile once.  A cluster of two CTAs splits the heads:
//   warp 0      TMA producer: the CTA's dK_h tiles (with their R_h boxes) into a ring, the B_h^T
//               boxes once the first tiles are on their way; each tile starts its walk over the
//               heads at a different head, so that the CTAs do not all read one head's columns
//               at once;
//   warp 1      TMEM owner; one thread issues dR_h = dK_h B_h (M = 128 tokens, N = r, K = d_h)
//               into r TMEM columns per head and, with dB folded in, dB_h's partial (M = d_h,
//               N = r, K = 128 tokens: the same dK_h tile read MN-major, R_h as a 16-column box
//               of 32-byte swizzle next to it in the stage) into r more columns per head;
//   warps 2..5  add every dK_h tile into fp32 registers (one token row per thread: G); after
//               each tile they store the previous head's dR row and fp32 dB partial row
//               ([H][tile][d_h][r], summed in tile order by the reduce kernel).  Each rank
//               finishes half of G's columns: it stages the other half of its partial G in its
//               idle ring and copies it in one bulk transfer into the peer's ring, then adds
//               the peer's half to its own and rounds the sum once.
// A ring slot is free once the MMAs (commit) and the four summing warps have read it.
namespace {

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cl_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Every thread of both CTAs: release its shared-memory writes, acquire the other CTA's.
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bulk copy from this CTA's shared memory into another CTA's (dst and bar: cluster addresses).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

template <int D_H>
struct DkCfg {
    static constexpr int NBOX = D_H / 64;
    static constexpr uint32_t TILE = NBOX * 16384u;  // one dK_h tile: 128 tokens x d_h
    static constexpr int STAGES = D_H == 128 ? 4 : 6;
    static constexpr int HALF = D_H / 2;             // G columns finished by each rank
    static constexpr int PITCH = HALF + 4;           // floats per row of a staged half of G
    static constexpr uint32_t GBYTES = 128u * PITCH * 4u;
    static constexpr uint32_t GOFF = (GBYTES + 1023u) & ~1023u;  // where the peer's half lands
};

}  // namespace

template <int D_H>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    dk_pass_kernel(const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmBT,
                   const __grid_constant__ CUtensorMap tmR, const DkArgs a) {
    using C = DkCfg<D_H>;
    constexpr int NBOX = C::NBOX, NST = C::STAGES, PITCH = C::PITCH, HALF = C::HALF;
    constexpr uint32_t TILE = C::TILE;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const int rank = (int)cl_rank();
    const int m0 = blockIdx.y * kTM;
    const int r = a.r;
    const int hpr = (a.H + 1) / 2;
    const int h0 = rank * hpr, nh = min(a.H - h0, hpr);
    const int hoff = (int)(blockIdx.y % (unsigned)nh);  // first head of this tile's walk
    const uint32_t BTB = (uint32_t)r * 128u;            // B^T box: r rows x 64 K
    const bool fdb = D_H == 128 && a.dBp != nullptr;     // dB folded in (r = 16)
    const uint32_t SST = TILE + (fdb ? 4096u : 0u);      // ring stage: dK_h tile [+ R_h box]
    const int dboff = hpr * r;                           // TMEM columns of the dB partials
    const uint32_t sRing = smem_u32(smem);
    const uint32_t sBT = sRing + NST * SST;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * SST + (size_t)hpr * NBOX * BTB);
    uint64_t* empty = full + NST;
    uint64_t* cfull = empty + NST;  // B^T boxes landed
    uint64_t* accf = cfull + 1;     // every MMA of this CTA has completed
    uint64_t* recv = accf + 1;      // the peer's half of G has landed in the ring
    // [2 NST] the MMAs of head i have completed (barrier i % 2 NST).  Head i's barrier completes
    // again only for head i + 2 NST, whose tile needs slot i % NST freed after head i + NST --
    // which the summing warps release only after draining head i (they drain head i after
    // summing head i + 1).  With NST barriers a slow drain could see head i + NST's completion
    // too and wait for a phase that never comes.
    uint64_t* mmad = recv + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mmad + 2 * NST);
    volatile int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 5);  // the MMA commit and the four summing warps
        }
        mbar_init(smem_u32(cfull), 1);
        mbar_init(smem_u32(accf), 1);
        mbar_init(smem_u32(recv), 1);
        for (int s = 0; s < 2 * NST; ++s) mbar_init(smem_u32(&mmad[s]), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    float g[D_H];  // this thread's token row of G (summing warps)
    if (warp == 0) {
        if (lane == 0) {
            const uint32_t cb = smem_u32(cfull);
            bool bt_issued = false;
            auto issue_bt = [&]() {
                mbar_arrive_expect_tx(cb, (uint32_t)nh * NBOX * BTB);
                for (int hh = 0; hh < nh; ++hh)
#pragma unroll
                    for (int j = 0; j < NBOX; ++j)
                        tma_load_2d(sBT + (hh * NBOX + j) * BTB, &tmBT, 64 * j, (h0 + hh) * r, cb);
                bt_issued = true;
            };
            int issued = 0;
            for (int i = 0; i < nh; ++i) {
                if (i == NST) issue_bt();  // the first tiles are on their way: now the B^T boxes
                const int s = i % NST, hh = (i + hoff) % nh;
                if ((i >= NST && !mbar_wait(smem_u32(&empty[s]), ((i / NST) - 1) & 1, a.status)) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                const uint32_t bar = smem_u32(&full[s]);
                mbar_arrive_expect_tx(bar, SST);
#pragma unroll
                for (int j = 0; j < NBOX; ++j)
                    tma_load_2d(sRing + s * SST + j * 16384, &tmdK, (h0 + hh) * D_H + 64 * j, m0, bar);
                if (fdb) tma_load_2d(sRing + s * SST + TILE, &tmR, a.rx0 + (h0 + hh) * r, m0, bar);
                issued = i + 1;
            }
            if (!bt_issued) issue_bt();
            mbar_wait(cb, 0, a.status);  // the B^T boxes have landed before the CTA can exit
            if (*abort_flag)             // as have the tiles in flight
                for (int k = max(0, issued - NST); k < issued; ++k)
                    mbar_wait(smem_u32(&full[k % NST]), (k / NST) & 1, a.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idR = idesc_bf16_f32(kTM, r);
            const uint32_t idB = idesc_bf16_f32(kTM, r) | (1u << 15) | (1u << 16);  // both MN-major
            bool ok = mbar_wait(smem_u32(cfull), 0, a.status);
            for (int i = 0; i < nh && ok; ++i) {
                const int s = i % NST, hh = (i + hoff) % nh;
                if (*abort_flag || !mbar_wait(smem_u32(&full[s]), (i / NST) & 1, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D_H / 16; ++kk) {
                    const int j = kk >> 2;
                    const uint32_t o = (kk & 3) * 32;
                    tc_mma_bf16(tmem + hh * r, kmaj(sRing + s * SST + j * 16384 + o),
                                kmaj(sBT + (hh * NBOX + j) * BTB + o), idR, kk != 0);
                }
                if (fdb)  // A = dK_h^T: 64-row blocks 16 KiB apart, 16 tokens (2 KiB) per K step
#pragma unroll
                    for (int kk = 0; kk < kTM / 16; ++kk)
                        tc_mma_bf16(tmem + dboff + hh * r, sdesc(sRing + s * SST + kk * 2048, 16384, 1024, 2),
                                    sdesc(sRing + s * SST + TILE + kk * 512, 16, 256, 6), idB, kk != 0);
                tc_commit(smem_u32(&empty[s]));
                tc_commit(smem_u32(&mmad[i % (2 * NST)]));
            }
            if (ok) tc_commit(smem_u32(accf));
            else *abort_flag = 1;
        }
    } else {
        // G: add each dK_h tile's row into fp32 registers; after each tile, store the previous
        // head's dR row (and dB partial row), whose MMAs have completed by then
        const int rl = (warp & 3) * 32 + lane;  // tile row = TMEM lane of this warp's quarter
        const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
        const int row = m0 + rl;
        auto drain = [&](int i) -> bool {
            const int hh = (i + hoff) % nh;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&mmad[i % (2 * NST)]), (i / (2 * NST)) & 1, a.status)))
                return false;
            tc_fence_after();
            uint16_t* grow = a.Gc + (size_t)row * a.ldg + D_H + (h0 + hh) * r;
            for (int c0 = 0; c0 < r; c0 += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + lanes + hh * r + c0, v);
                if (row < a.n) {
                    uint4 p0, p1;
                    p0.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
                    p0.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
                    p0.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
                    p0.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
                    p1.x = pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9]));
                    p1.y = pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11]));
                    p1.z = pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13]));
                    p1.w = pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15]));
                    reinterpret_cast<uint4*>(grow + c0)[0] = p0;
                    reinterpret_cast<uint4*>(grow + c0)[1] = p1;
                }
            }
            if (fdb) {
                // this tile's dB_h partial: TMEM lane = d_h row, r = 16 columns
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + lanes + dboff + hh * r, v);
                float4* dst = reinterpret_cast<float4*>(
                    a.dBp + ((((size_t)(h0 + hh) * gridDim.y + blockIdx.y) * kTM + rl) * r));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                         __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            return true;
        };
#pragma unroll
        for (int c = 0; c < D_H; ++c) g[c] = 0.f;
        bool ok = true;
        for (int i = 0; i < nh; ++i) {
            const int s = i % NST;
            ok = ok && !*abort_flag && mbar_wait(smem_u32(&full[s]), (i / NST) & 1, a.status);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            const uint8_t* tile = smem + s * SST + rl * 128;
#pragma unroll
            for (int j = 0; j < NBOX; ++j)
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 v = *reinterpret_cast<const uint4*>(tile + j * 16384 + ((c8 ^ (rl & 7)) << 4));
                    float* gg = g + j * 64 + c8 * 8;
                    gg[0] += bf16lo(v.x); gg[1] += bf16hi(v.x); gg[2] += bf16lo(v.y); gg[3] += bf16hi(v.y);
                    gg[4] += bf16lo(v.z); gg[5] += bf16hi(v.z); gg[6] += bf16lo(v.w); gg[7] += bf16hi(v.w);
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            if (i > 0 && !drain(i - 1)) {
                ok = false;
                break;
            }
        }
        if (ok && nh > 0) ok = drain(nh - 1);
        ok = ok && mbar_wait(smem_u32(accf), 0, a.status);
        if (!__all_sync(0xffffffffu, ok) && lane == 0) *abort_flag = 1;
        tc_fence_after();
        // stage the half of the partial G that the peer finishes (rank 0 finishes columns
        // [0, d_h / 2), rank 1 the rest) in this CTA's idle ring
        float* dst = reinterpret_cast<float*>(smem) + (size_t)rl * PITCH;
        if (rank == 0) {
#pragma unroll
            for (int c = 0; c < HALF; c += 4)
                *reinterpret_cast<float4*>(dst + c) = make_float4(g[HALF + c], g[HALF + c + 1], g[HALF + c + 2], g[HALF + c + 3]);
        } else {
#pragma unroll
            for (int c = 0; c < HALF; c += 4)
                *reinterpret_cast<float4*>(dst + c) = make_float4(g[c], g[c + 1], g[c + 2], g[c + 3]);
        }
        fence_proxy_async_smem();  // generic writes, before the bulk copy reads them
        if (threadIdx.x == 64) mbar_arrive_expect_tx(smem_u32(recv), C::GBYTES);
    }
    // Barrier 1: both rings are idle (every stage consumed, every MMA complete), each rank's half
    // for the peer is staged and each rank expects the peer's.
    __syncwarp();
    cl_sync();
    if (warp >= 2) {
        const int rl = (warp & 3) * 32 + lane;
        const int row = m0 + rl;
        const bool ok = !*abort_flag;
        if (threadIdx.x == 64 && ok)
            bulk_copy_to_peer(cl_map(sRing + C::GOFF, rank ^ 1), sRing, C::GBYTES, cl_map(smem_u32(recv), rank ^ 1));
        if (ok && mbar_wait(smem_u32(recv), 0, a.status) && row < a.n) {
            const float* rv = reinterpret_cast<const float*>(smem + C::GOFF) + (size_t)rl * PITCH;
            uint16_t* grow = a.Gc + (size_t)row * a.ldg + rank * HALF;
            auto finish = [&](const float* mine) {
#pragma unroll
                for (int c = 0; c < HALF; c += 8) {
                    const float4 x0 = *reinterpret_cast<const float4*>(rv + c);
                    const float4 x1 = *reinterpret_cast<const float4*>(rv + c + 4);
                    uint4 pk;
                    pk.x = pack_bf16x2(mine[c] + x0.x, mine[c + 1] + x0.y);
                    pk.y = pack_bf16x2(mine[c + 2] + x0.z, mine[c + 3] + x0.w);
                    pk.z = pack_bf16x2(mine[c + 4] + x1.x, mine[c + 5] + x1.y);
                    pk.w = pack_bf16x2(mine[c + 6] + x1.z, mine[c + 7] + x1.w);
                    *reinterpret_cast<uint4*>(grow + c) = pk;
                }
            };
            if (rank == 0) finish(g);
            else finish(g + HALF);
        }
    }
    // Barrier 2: both ranks have received the peer's copy, so the staging may go
    __syncwarp();
    cl_sync();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// BT[h][j][e] = B[h][e][j]: the residual factors as K-major [r][d_h] blocks.
__global__ void __launch_bounds__(256) bt_kernel(const uint16_t* B, uint16_t* BT, int H, int d_h, int r) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= H * r * d_h) return;
    const int h = idx / (r * d_h), rem = idx % (r * d_h);
    const int j = rem / d_h, e = rem % d_h;
    BT[idx] = B[((size_t)h * d_h + e) * r + j];
}

template <int D_H>
static size_t dk_smem(int H, int r, bool fdb) {
    return (size_t)DkCfg<D_H>::STAGES * (DkCfg<D_H>::TILE + (fdb ? 4096 : 0)) +
           (size_t)((H + 1) / 2) * DkCfg<D_H>::NBOX * r * 128 + 256 + 1024;
}

bool dk_pass_supported(int H, int d_h, int r) {
    if (H < 2 || !(d_h == 64 || d_h == 128) || !(r == 16 || r == 32) || ((H + 1) / 2) * r > 512) return false;
    return (d_h == 64 ? dk_smem<64>(H, r, false) : dk_smem<128>(H, r, false)) <= kTSmemMax;
}

bool dk_pass_folds_dB(int H, int d_h, int r) {
    return dk_pass_supported(H, d_h, r) && d_h == 128 && r == 16 && 2 * ((H + 1) / 2) * r <= 512 &&
           dk_smem<128>(H, r, true) <= kTSmemMax;
}

template <int D_H>
static cudaError_t launch_dk_t(const CUtensorMap& tdK, const CUtensorMap& tBT, const CUtensorMap& tR, const DkArgs& a,
                               cudaStream_t stream) {
    // the staged half of G and the peer's half fit in the ring
    static_assert((size_t)DkCfg<D_H>::STAGES * DkCfg<D_H>::TILE >= DkCfg<D_H>::GOFF + DkCfg<D_H>::GBYTES, "ring");
    // at least 120 KiB, so that one CTA runs per SM: each allocates all 512 TMEM columns, and a
    // second resident CTA would wait in its allocation for one that waits on its cluster peer
    const size_t need = dk_smem<D_H>(a.H, a.r, a.dBp != nullptr), smem = need > 122880 ? need : 122880;
    auto kern = dk_pass_kernel<D_H>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(2, (a.n + kTM - 1) / kTM), 192, smem, stream>>>(tdK, tBT, tR, a);
    return cudaGetLastError();
}

cudaError_t launch_dk_pass(const CUtensorMap& tdK, const CUtensorMap& tBT, const CUtensorMap& tR, const uint16_t* B,
                           uint16_t* BT, const DkArgs& a, cudaStream_t stream) {
    if (!dk_pass_supported(a.H, a.d_h, a.r) || (a.dBp && !dk_pass_folds_dB(a.H, a.d_h, a.r)))
        return cudaErrorInvalidValue;
    const int tot = a.H * a.r * a.d_h;
    bt_kernel<<<(tot + 255) / 256, 256, 0, stream>>>(B, BT, a.H, a.d_h, a.r);
    return a.d_h == 64 ? launch_dk_t<64>(tdK, tBT, tR, a, stream) : launch_dk_t<128>(tdK, tBT, tR, a, stream);
}

// G[t][e] = sum_h dK[t][h][e] (fp32, heads in order), eight columns per thread.
__global__ void __launch_bounds__(256) head_sum_kernel(const uint16_t* dK, uint16_t* Gc, int n, int H, int d_h,
                                                       int ldg) {
    const int per_row = d_h / 8;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)n * per_row) return;
    const int t = (int)(idx / per_row), c = (int)(idx % per_row) * 8;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const uint16_t* src = dK + (size_t)t * H * d_h + c;
    for (int h = 0; h < H; ++h) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(src + (size_t)h * d_h));
        f[0] += bf16lo(x.x); f[1] += bf16hi(x.x); f[2] += bf16lo(x.y); f[3] += bf16hi(x.y);
        f[4] += bf16lo(x.z); f[5] += bf16hi(x.z); f[6] += bf16lo(x.w); f[7] += bf16hi(x.w);
    }
    uint4 pk;
    pk.x = pack_bf16x2(f[0], f[1]);
    pk.y = pack_bf16x2(f[2], f[3]);
    pk.z = pack_bf16x2(f[4], f[5]);
    pk.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(Gc + (size_t)t * ldg + c) = pk;
}

// dB[h][e][j] = sum over ks of P[h][ks][e][j], bf16 (partials [H][ks][128][pw]).  A block of 256
// threads covers 64 outputs of four consecutive j each; its four thread groups sum interleaved
// quarters of the partials (sixteen loads in flight per thread), then group 0 adds the four
// sums in group order -- a fixed order, so the result does not depend on timing.
__global__ void __launch_bounds__(256) dB_reduce_kernel(const float* P, uint16_t* dB, int H, int ksplit, int d_h,
                                                        int r, int pw) {
    __shared__ float4 part[4][64];
    const int r4 = r / 4;
    const int grp = threadIdx.x >> 6, t = threadIdx.x & 63;
    const long long idx = (long long)blockIdx.x * 64 + t;
    const bool live = idx < (long long)H * d_h * r4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int h = 0, e = 0, j = 0;
    if (live) {
        h = (int)(idx / ((long long)d_h * r4));
        const int rem = (int)(idx % ((long long)d_h * r4));
        e = rem / r4;
        j = (rem % r4) * 4;
        const float4* src = reinterpret_cast<const float4*>(P + (((size_t)h * ksplit) * kTM + e) * pw + j);
        const size_t stride = (size_t)kTM * pw / 4;  // float4s between consecutive partials
        for (int k0 = grp; k0 < ksplit; k0 += 4 * 16) {
            float4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int k = k0 + 4 * u;
                v[u] = k < ksplit ? __ldg(src + (size_t)k * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                acc.x += v[u].x;
                acc.y += v[u].y;
                acc.z += v[u].z;
                acc.w += v[u].w;
            }
        }
    }
    part[grp][t] = acc;
    __syncthreads();
    if (grp == 0 && live) {
        float4 s4 = part[0][t];
#pragma unroll
        for (int g = 1; g < 4; ++g) {
            s4.x += part[g][t].x;
            s4.y += part[g][t].y;
            s4.z += part[g][t].z;
            s4.w += part[g][t].w;
        }
        uint2 o;
        o.x = pack_bf16x2(s4.x, s4.y);
        o.y = pack_bf16x2(s4.z, s4.w);
        *reinterpret_cast<uint2*>(dB + ((size_t)h * d_h + e) * r + j) = o;
    }
}

static int tgemm_tiles(const GemmArgs& g, int bn) {
    return ((g.N + bn - 1) / bn) * ((g.M + kTM - 1) / kTM) * g.nbatch * g.ksplit;
}

// One launch over p.ngroups products (their tiles in order: group 0 first); dynamic: items after
// each CTA's first come from the queue at p.ctr, which must be zero at launch.
static cudaError_t tgemm_launch(TGemmParams& p, int bn, bool out_f32, bool dynamic, cudaStream_t stream) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    for (int i = 0; i < p.ngroups; ++i) {
        const GemmArgs& g = p.g[i];
        if (g.kfix % kTK != 0 || (g.kfix > 0 && (g.a_mn || g.b_mn || i > 0))) return cudaErrorInvalidValue;
    }
    p.tiles0 = tgemm_tiles(p.g[0], bn);
    p.total = p.tiles0 + (p.ngroups > 1 ? tgemm_tiles(p.g[1], bn) : 0);
    if (p.total == 0) return cudaSuccess;
    if (!dynamic) p.ctr = nullptr;
    const dim3 grid((unsigned)(p.total < sms ? p.total : sms));
#define LRKV_TG(OF, NB, GR)                                                                                     \
    if (out_f32 == OF && bn == NB && (p.ngroups > 1) == GR) {                                                   \
        auto kern = tgemm_kernel<OF, NB, GR>;                                                                   \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TCfg<NB>::SMEM); \
        if (e != cudaSuccess) return e;                                                                         \
        kern<<<grid, 192, TCfg<NB>::SMEM, stream>>>(p);                                                         \
        return cudaGetLastError();                                                                              \
    }
    LRKV_TG(false, 128, false)  // expansion, dR
    LRKV_TG(false, 160, false)  // Y
    LRKV_TG(false, 256, false)  // dW_T or dX alone
    LRKV_TG(false, 256, true)   // dW_T and dX together
    LRKV_TG(true, 64, false)    // dB partials
#undef LRKV_TG
    return cudaErrorInvalidValue;
}

cudaError_t launch_tgemm(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tB2, const CUtensorMap& tC,
                         const GemmArgs& g, int bn, bool out_f32, cudaStream_t stream) {
    TGemmParams p;
    memset(&p, 0, sizeof(p));
    p.A[0] = p.A[1] = tA;
    p.B[0] = p.B[1] = tB;
    p.C[0] = p.C[1] = tC;
    p.B2 = tB2;
    p.g[0] = p.g[1] = g;
    p.ngroups = 1;
    return tgemm_launch(p, bn, out_f32, false, stream);
}

cudaError_t launch_tgemm2(const CUtensorMap* tA, const CUtensorMap* tB, const CUtensorMap* tC, const GemmArgs* g, int bn,
                          int* ctr, cudaStream_t stream) {
    TGemmParams p;
    memset(&p, 0, sizeof(p));
    for (int i = 0; i < 2; ++i) {
        p.A[i] = tA[i];
        p.B[i] = tB[i];
        p.C[i] = tC[i];
        p.g[i] = g[i];
    }
    p.B2 = tB[0];
    p.ngroups = 2;
    p.ctr = ctr;
    cudaError_t e = cudaMemsetAsync(ctr, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    return tgemm_launch(p, bn, false, true, stream);
}

cudaError_t launch_head_sum(const uint16_t* dK, uint16_t* Gc, int n, int H, int d_h, int ldg, cudaStream_t stream) {
    const long long total = (long long)n * (d_h / 8);
    head_sum_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(dK, Gc, n, H, d_h, ldg);
    return cudaGetLastError();
}

cudaError_t launch_dB_reduce(const float* P, uint16_t* dB, int H, int ksplit, int d_h, int r, int pw,
                             cudaStream_t stream) {
    if (r % 4 != 0 || pw % 4 != 0) return cudaErrorInvalidValue;
    const long long total = (long long)H * d_h * (r / 4);
    dB_reduce_kernel<<<(unsigned)((total + 63) / 64), 256, 0, stream>>>(P, dB, H, ksplit, d_h, r, pw);
    return cudaGetLastError();
}

}  // namespace lrkv
