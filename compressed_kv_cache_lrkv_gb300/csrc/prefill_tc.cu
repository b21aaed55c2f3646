// prefill_tc.cu -- causal chunked prefill on the 5th-generation tensor cores
// ("Low-Rank Key Value Attention", Eqs. (6)-(7) with the causal mask of the
// softmax frame), for d_h = 64 or 128 and r = 16, and for d_h = 128 with the decoupled
// positional key (d_rope = 64: key rows [s^K | k^R], queries [q | q^R]).
//
// One CTA = 128 queries of one (sequence, head); key tiles of 128 tokens (two
// cache pages).  Per tile j:
//   S_j  = [Q | Q~] . [s^K | z^K_h]^T     tcgen05.mma M=128 N=128, K = 128 + 16,
//                                          fp32 in TMEM (two S buffers)
//   P_j  = exp2(S_j * scale * log2 e - m) bf16, written back into the first 64 TMEM
//          columns of S_j's own buffer
//   O_s += P_j . s^V (N = 128),  O_z += P_j . z^V_h (N = 16)   in TMEM, A operand P_j
//          read from TMEM
// with Q~ = Q . B_h^K computed on the tensor cores in the prologue.  After the last
// tile O_s += O_z . (B_h^V)^T runs as two kind::tf32 MMAs (A = O_z straight from TMEM,
// B = B_h^V widened to fp32 in shared memory), so the epilogue is out = O_s / l.  Warp roles: warp 0 key-tile TMA
// producer (3-stage ring), warp 6 value-tile TMA producer (2-stage ring), warp 1
// score-MMA issuer and TMEM owner, warp 7 P.V-MMA issuer, warps 2..5 softmax /
// epilogue (one query row per thread, TMEM lane quarter = warp % 4).
// The running max is only raised (and O rescaled in TMEM) when a row's max grows
// by more than 2^8, so most tiles need no O round trip.  Key rows past the
// context are zero-filled (TMA out-of-bounds fill, or cleared in shared memory)
// so masked tokens cannot inject NaN through 0 * garbage.
// With a positional key the shared logits run over D_K = d_h + 64 columns and the key ring
// has two stages (its stages grow by 16 KB); Q~ then lives in TMEM as the A operand of its
// MMA instead of in shared memory, B^K is staged in the second value stage (the value
// producer fills that stage only after the Q~ MMA has read it) and B^V, at the end, in the
// first key stage.
#include <type_traits>

#include "kernels.h"
#include "lrkv_internal.cuh"

namespace lrkv {

namespace {

constexpr int kBM = 128, kBN = 128;
constexpr int kVStages = 2;
// Shared-memory layout for d_h = D_H and a positional key of D_R columns (the tiles are blocks
// of 64 columns; D_K = D_H + D_R):
//   Q    [128 q][D_K] K-major, 128B swizzle
//   Q~   [128 q][16] K-major, 32B swizzle (no positional key; with one, Q~ sits in TMEM)
//   B^K  [D_H d][16] MN-major (B operand of Q~), 32B swizzle
//   B^V  as fp32 for the final tf32 MMA: [D_H d][16 j], K-major without swizzle -- 8 x
//        4-element core matrices, element (d, j) at (d / 8) * 512 + (j / 4) * 128 + (d % 8) * 16
//        + (j % 4) * 4.  Without a positional key it takes the place of B^K (and the 4 KB
//        after it) once Q~ is computed; with one it goes into key stage 0 after the last S MMA.
//   key ring (3 stages, 2 with a positional key: [s^K | k^R] [128 keys][D_K] K-major 128B
//   swizzle, then z^K_h [128][16] 32B swizzle) and value ring (2 stages: s^V [128][D_H],
//   z^V_h, same layouts, read MN-major); with a positional key B^K sits in value stage 1.
template <int D_H, int D_R>
struct PfLayout {
    static constexpr bool ROPE = D_R > 0;
    static constexpr int D_K = D_H + D_R;
    static constexpr int KST = ROPE ? 2 : 3;  // key ring stages
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t Q_BYTES = 128 * D_K * 2;
    static constexpr uint32_t K_Z = 128 * D_K * 2, K_BYTES = K_Z + 4096;  // key stage: [s^K | k^R], z^K_h
    static constexpr uint32_t V_Z = 128 * D_H * 2, V_BYTES = V_Z + 4096;  // value stage: s^V, z^V_h
    static constexpr uint32_t OFF_QT = Q_BYTES;
    static constexpr uint32_t OFF_K = ROPE ? Q_BYTES : OFF_QT + 4096 + D_H * 64;
    static constexpr uint32_t OFF_V = OFF_K + KST * K_BYTES;
    static constexpr uint32_t OFF_BK = ROPE ? OFF_V + V_BYTES : OFF_QT + 4096;
    static constexpr uint32_t OFF_BVF = ROPE ? OFF_K : OFF_BK;
    static constexpr uint32_t OFF_BAR = OFF_V + kVStages * V_BYTES;
    static constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
    static_assert(OFF_K % 1024 == 0 && K_BYTES % 1024 == 0 && V_BYTES % 1024 == 0 && OFF_BK % 1024 == 0,
                  "swizzled TMA tiles start 1024-aligned");
    static_assert(D_H * 64 <= (ROPE ? K_BYTES : 8192), "B^V (fp32) fits its area");
    static_assert(SMEM <= 232448, "fits one CTA's opt-in shared memory");
};
// TMEM columns: S buffers, O_s, O_z, Q~ (fp32 from its MMA) and, with a positional key, Q~ as
// bf16 pairs (the A operand of its MMA).
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_OS = 256, TM_OZ = 384, TM_QTB = 400, TM_QT = 448, TM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ uint64_t kdesc128(uint32_t a) { return sdesc(a, 16, 1024, 2); }
__device__ __forceinline__ uint64_t kdesc32(uint32_t a) { return sdesc(a, 16, 256, 6); }
__device__ __forceinline__ uint64_t mndesc128(uint32_t a) { return sdesc(a, 16384, 1024, 2); }
__device__ __forceinline__ uint64_t mndesc32(uint32_t a) { return sdesc(a, 16, 256, 6); }

// Three-input f32 maximum (sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 32 lanes x 8 consecutive 32-bit columns, register -> TMEM.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, uint32_t* status) {
    const bool ok = mbar_wait(bar, parity, status);
    return __all_sync(0xffffffffu, ok);
}

}  // namespace

constexpr int kThreads = 256;

// FUSED: absorbed weights -- Q~ arrives from the caller (TMA into the Q~ tile, no absorption
// MMA) and the epilogue returns [O_s | O_z] / l (no B^V MMA).
template <int D_H, int D_R, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillMaps m, const PrefillArgs a) {
    constexpr int R = 16;
    constexpr int OW = FUSED ? D_H + R : D_H;  // output row width
    using Lay = PfLayout<D_H, D_R>;
    constexpr bool ROPE = Lay::ROPE;
    static_assert(!(ROPE && FUSED), "absorbed weights with a positional key run on the warp-level kernel");
    constexpr int D_K = Lay::D_K, KST = Lay::KST;
    constexpr int NBK = D_K / 64, NBV = D_H / 64;  // 64-column blocks of a key / value row
    constexpr uint32_t OFF_Q = Lay::OFF_Q, OFF_QT = Lay::OFF_QT, OFF_BK = Lay::OFF_BK, OFF_BVF = Lay::OFF_BVF;
    constexpr uint32_t K_Z = Lay::K_Z, K_BYTES = Lay::K_BYTES, V_Z = Lay::V_Z, V_BYTES = Lay::V_BYTES;
    constexpr uint32_t OFF_K = Lay::OFF_K, OFF_V = Lay::OFF_V, OFF_BAR = Lay::OFF_BAR;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t S0 = smem_u32(smem);

    const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;  // heavy query tiles first
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Tq = a.Tq, H = a.H;
    const int qs = a.q_start[b];
    const int ctx = qs + Tq;
    const int q0 = qt * kBM;
    auto out_row = [&](int i) { return a.out + (((size_t)b * Tq + i) * H + h) * OW; };
    if (qs < 0 || ctx > a.max_pages * kBlockSize) {
        if (threadIdx.x == 0 && qt == 0 && h == 0) set_status(a.status, LRKV_DEV_BAD_SEQLEN);
        for (int idx = threadIdx.x; idx < kBM * OW; idx += blockDim.x) {
            const int i = q0 + idx / OW;
            if (i < Tq) out_row(i)[idx % OW] = 0;
        }
        return;
    }
    const int last_row = min(q0 + kBM - 1, Tq - 1);
    const int nt = (qs + last_row) / kBN + 1;  // key tiles this CTA needs

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* qt_mma = bars + 1;
    uint64_t* qt_ready = bars + 2;
    uint64_t* s_full = bars + 3;    // [2]
    uint64_t* p_full = bars + 5;
    // o_done[j % 2]: P_j . V_j complete.  Softmax waits on it only before rescaling O (rare),
    // so it may skip phases; two barriers by tile parity keep that safe: o_done[j % 2] cannot
    // complete its next phase (P_{j+2} . V_{j+2}) before softmax has passed tile j + 2.
    uint64_t* o_done = bars + 23;   // [2]
    uint64_t* fin_done = bars + 25;  // O_s += O_z . B^V^T complete
    uint64_t* mma_drain = bars + 7;  // all MMAs of the CTA complete
    uint64_t* k_full = bars + 8;    // [3] s^K, z^K of a key tile landed
    uint64_t* k_empty = bars + 11;  // [3] S MMA done with them
    uint64_t* v_full = bars + 14;   // [2] s^V, z^V landed
    uint64_t* v_empty = bars + 16;  // [2] P.V MMA done with them
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
    volatile int* abort_flag = reinterpret_cast<int*>(bars + 19);
    uint64_t* s_free = bars + 20;    // [2] P_j . V_j done: S buffer j % 2 may take S_{j+2}
    uint64_t* pv_drain = bars + 22;  // all P.V MMAs complete
    uint64_t* bvf_ready = bars + 26;  // positional key: B^V (fp32) written into key stage 0
    auto B = [&](uint64_t* p) { return smem_u32(p); };
    // The abort flag is read warp-uniformly: a warp whose lanes saw different values would
    // reach its later warp-wide votes and shuffles with only some of its lanes.
    auto aborted = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0); };

    if (threadIdx.x == 0) {
        mbar_init(B(q_full), 1);
        mbar_init(B(qt_mma), 1);
        mbar_init(B(qt_ready), 128);
        for (int i = 0; i < KST; ++i) {
            mbar_init(B(k_full + i), 1);
            mbar_init(B(k_empty + i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(B(v_full + i), 1);
            mbar_init(B(v_empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(B(s_full + i), 1);
        mbar_init(B(p_full), 128);
        for (int i = 0; i < 2; ++i) mbar_init(B(o_done + i), 1);
        mbar_init(B(fin_done), 1);
        mbar_init(B(bvf_ready), 128);
        mbar_init(B(mma_drain), 1);
        mbar_init(B(pv_drain), 1);
        for (int i = 0; i < 2; ++i) mbar_init(B(s_free + i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == 6) {
        // ---------------------------------------------------------------- TMA producers
        // Warp 0 streams key tiles (s^K, z^K_h) into the 3-stage key ring, warp 6 value
        // tiles (s^V, z^V_h) into the 2-stage value ring; each waits only on its own ring.
        // Physical rows of this sequence's pages sit in registers, 32 pages per batch (lane
        // i holds page 32 * batch + i), the next batch fetched one batch ahead, so no
        // dependent global load sits between two tiles' copies.
        const bool keys = warp == 0;
        const int oob_row = a.num_blocks * kBlockSize;  // whole box out of bounds -> zero fill
        const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
        auto fetch = [&](int batch) {
            const int page = batch * 32 + lane;
            int row = oob_row;
            if (page < a.max_pages && page * kBlockSize < ctx) {
                const int blk = bt[page];
                if (blk >= 0 && blk < a.num_blocks)
                    row = blk * kBlockSize;
                else
                    set_status(a.status, LRKV_DEV_BAD_BLOCK);
            }
            return row;
        };
        if (keys && lane == 0) {
            mbar_arrive_expect_tx(B(q_full), 128 * D_K * 2 + (FUSED ? 128 * R * 2 : D_H * R * 2));
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk) tma_load_2d(S0 + OFF_Q + bk * 16384, &m.q, h * D_K + 64 * bk, b * Tq + q0, B(q_full));
            if (FUSED)
                tma_load_2d(S0 + OFF_QT, &m.qt, h * R, b * Tq + q0, B(q_full));
            else
                tma_load_2d(S0 + OFF_BK, &m.BK, 0, h * D_H, B(q_full));
        }
        const int depth = keys ? KST : kVStages;
        const uint32_t stage_bytes = keys ? K_BYTES : V_BYTES, zoff = keys ? K_Z : V_Z;
        const int nblk = keys ? NBK : NBV;
        uint64_t* full = keys ? k_full : v_full;
        uint64_t* empty = keys ? k_empty : v_empty;
        const CUtensorMap* ms = keys ? &m.sK : &m.sV;
        const CUtensorMap* mz = keys ? &m.zK : &m.zV;
        const uint32_t ring = S0 + (keys ? OFF_K : OFF_V);
        int cur = fetch(0), nxt = fetch(1);
        int issued = 0;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            if (j > 0 && (j & 15) == 0) {  // pages 2j, 2j+1 start a new batch of 32
                cur = nxt;
                nxt = fetch((j >> 4) + 1);
            }
            const int row0 = __shfl_sync(0xffffffffu, cur, (2 * j) & 31);
            const int row1 = __shfl_sync(0xffffffffu, cur, (2 * j + 1) & 31);
            const int st = j % depth;
            if (j >= depth && !wait_all(B(empty + st), (j / depth - 1) & 1, a.status)) {
                ok = false;
                break;
            }
            // with a positional key, value stage 1 holds B^K until the Q~ MMA has read it
            if (ROPE && !keys && j == 1 && !wait_all(B(qt_mma), 0, a.status)) {
                ok = false;
                break;
            }
            if (aborted()) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t base = ring + st * stage_bytes, bar = B(full + st);
                mbar_arrive_expect_tx(bar, stage_bytes);
                for (int p = 0; p < 2; ++p) {
                    const int row = p ? row1 : row0;
                    for (int bk = 0; bk < nblk; ++bk) tma_load_2d(base + bk * 16384 + p * 8192, ms, 64 * bk, row, bar);
                    tma_load_2d(base + zoff + p * 2048, mz, h * R, row, bar);
                }
            }
            __syncwarp();
            issued = j + 1;
        }
        if (!ok) {
            *abort_flag = 1;
            // let this ring's copies still in flight land before the CTA exits
            for (int k = max(0, issued - depth); k < issued; ++k) wait_all(B(full + k % depth), (k / depth) & 1, a.status);
        }
    } else if (warp == 1 || warp == 7) {
        // ---------------------------------------------------------------- MMA issuers
        // tcgen05.mma issue blocks once the tensor pipe's queue is full, so one issuing
        // thread that also waits on barriers leaves the pipe idle between its bursts.  Two
        // warps issue instead: warp 1 the score MMAs (Q~ in the prologue, then S_j), warp 7
        // the P.V MMAs.  Each runs converged and lets one elected lane issue its tcgen05
        // instructions and commits.  Descriptors are built once and advanced by adding
        // (byte offset >> 4) to their start-address field; the tile loops are unrolled over
        // the ring stages (6 = lcm of the 3 key stages and 2 S buffers; 2 value stages) so
        // every operand of every MMA is loop-invariant -- operands that change from tile
        // to tile cost a register-to-uniform move per MMA and halve the issue rate.
        constexpr uint32_t id_S = idesc_bf16_f32(128, 128);
        constexpr uint32_t id_QT = idesc_bf16_f32(128, 16) | (1u << 16);
        constexpr uint32_t id_PVs = idesc_bf16_f32(128, D_H) | (1u << 16);
        constexpr uint32_t id_PVz = idesc_bf16_f32(128, 16) | (1u << 16);
        constexpr uint64_t kKStage = K_BYTES >> 4, kVStage = V_BYTES >> 4;
        bool ok = true;
        if (warp == 1) {
            const uint64_t dQ = kdesc128(S0 + OFF_Q), dQT = kdesc32(S0 + OFF_QT), dBK = mndesc32(S0 + OFF_BK);
            const uint64_t dSK = kdesc128(S0 + OFF_K), dZK = kdesc32(S0 + OFF_K + K_Z);
            // K-step kk of a K-major 128-byte-swizzled [rows][128] tile: 64-column block kk/4, 32 bytes in.
            auto kstep = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
            ok = wait_all(B(q_full), 0, a.status);
            if (!FUSED) {
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D_H / 16; ++kk)
                        if (elect_one_sync())
                            tc_mma_bf16(tmem + TM_QT, dQ + kstep(kk), dBK + (kk * 512 >> 4), id_QT, kk > 0);
                }
                if (elect_one_sync()) tc_commit(B(qt_mma));
                __syncwarp();
                ok = ok && wait_all(B(qt_ready), 0, a.status);
            }
            auto s_tile = [&](int jj, auto U) -> bool {
                constexpr int st = decltype(U)::value % KST, sb = decltype(U)::value & 1;
                // S buffer sb still holds P_{jj-2} until P_{jj-2} . V_{jj-2} has completed
                if (aborted() || !wait_all(B(k_full + st), (jj / KST) & 1, a.status) ||
                    (jj >= 2 && !wait_all(B(s_free + sb), ((jj >> 1) - 1) & 1, a.status)))
                    return false;
                tc_fence_after();
                constexpr uint64_t so = st * kKStage;
                const uint32_t d = tmem + (sb ? TM_S1 : TM_S0);
#pragma unroll
                for (int kk = 0; kk < D_K / 16; ++kk)
                    if (elect_one_sync()) tc_mma_bf16(d, dQ + kstep(kk), dSK + so + kstep(kk), id_S, kk > 0);
                if (elect_one_sync()) {
                    if (ROPE)
                        tc_mma_bf16_ts(d, tmem + TM_QTB, dZK + so, id_S, 1);
                    else
                        tc_mma_bf16(d, dQT, dZK + so, id_S, 1);
                    tc_commit(B(s_full + sb));
                    tc_commit(B(k_empty + st));
                }
                __syncwarp();
                return true;
            };
            using I0 = std::integral_constant<int, 0>;
            using I1 = std::integral_constant<int, 1>;
            using I2 = std::integral_constant<int, 2>;
            using I3 = std::integral_constant<int, 3>;
            using I4 = std::integral_constant<int, 4>;
            using I5 = std::integral_constant<int, 5>;
            for (int jj = 0; jj < nt && ok; jj += 6) {
                ok = s_tile(jj, I0{});
                if (ok && jj + 1 < nt) ok = s_tile(jj + 1, I1{});
                if (ok && jj + 2 < nt) ok = s_tile(jj + 2, I2{});
                if (ok && jj + 3 < nt) ok = s_tile(jj + 3, I3{});
                if (ok && jj + 4 < nt) ok = s_tile(jj + 4, I4{});
                if (ok && jj + 5 < nt) ok = s_tile(jj + 5, I5{});
            }
            if (!ok) *abort_flag = 1;
            // Every MMA this warp issued has finished before the CTA tears TMEM down.
            if (elect_one_sync()) tc_commit(B(mma_drain));
            __syncwarp();
            wait_all(B(mma_drain), 0, a.status);
        } else {
            const uint64_t dSV = mndesc128(S0 + OFF_V), dZV = mndesc32(S0 + OFF_V + V_Z);
            auto pv_tile = [&](int j, auto PAR) -> bool {
                constexpr int vs = decltype(PAR)::value;  // value stage = S buffer = j % 2
                if (aborted() || !wait_all(B(p_full), j & 1, a.status) ||
                    !wait_all(B(v_full + vs), (j >> 1) & 1, a.status))
                    return false;
                tc_fence_after();
                constexpr uint64_t so = vs * kVStage;
                const uint32_t pt = tmem + (vs ? TM_S1 : TM_S0);  // P_j over S_j's columns
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    if (elect_one_sync()) {
                        tc_mma_bf16_ts(tmem + TM_OS, pt + kk * 8, dSV + so + (kk * 2048 >> 4), id_PVs, (j | kk) != 0);
                        tc_mma_bf16_ts(tmem + TM_OZ, pt + kk * 8, dZV + so + (kk * 512 >> 4), id_PVz, (j | kk) != 0);
                    }
                }
                if (elect_one_sync()) {
                    tc_commit(B(o_done + vs));
                    tc_commit(B(v_empty + vs));
                    tc_commit(B(s_free + vs));
                }
                __syncwarp();
                return true;
            };
            for (int j = 0; j < nt && ok; j += 2) {
                ok = pv_tile(j, std::integral_constant<int, 0>{});
                if (ok && j + 1 < nt) ok = pv_tile(j + 1, std::integral_constant<int, 1>{});
            }
            // O_s += O_z . (B_h^V)^T.  O_z is read as an MMA operand, so its last
            // accumulation must have completed first.
            ok = ok && wait_all(B(o_done + ((nt - 1) & 1)), ((nt - 1) >> 1) & 1, a.status);
            if (ROPE) ok = ok && wait_all(B(bvf_ready), 0, a.status);  // B^V in key stage 0
            if (ok && FUSED) {  // [O_s | O_z] leave as they are: fin_done only marks them complete
                if (elect_one_sync()) tc_commit(B(fin_done));
                __syncwarp();
            } else if (ok) {
                constexpr uint32_t id_fin = idesc_tf32_f32(128, D_H);
                const uint64_t dBV = sdesc(S0 + OFF_BVF, 128, 512, 0);
                tc_fence_after();
                if (elect_one_sync()) {
                    tc_mma_tf32_ts(tmem + TM_OS, tmem + TM_OZ, dBV, id_fin, 1);
                    tc_mma_tf32_ts(tmem + TM_OS, tmem + TM_OZ + 8, dBV + (256 >> 4), id_fin, 1);
                    tc_commit(B(fin_done));
                }
                __syncwarp();
            }
            if (!ok) *abort_flag = 1;
            if (elect_one_sync()) tc_commit(B(pv_drain));
            __syncwarp();
            wait_all(B(pv_drain), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- softmax / epilogue
        const int qq = warp & 3;
        const int row = qq * 32 + lane;              // query row within the tile = TMEM lane
        const uint32_t tl = (uint32_t)(qq * 32) << 16;
        const int st_tid = threadIdx.x - 64;         // 0..127
        // B_h^V widened to fp32 for the final tf32 MMA: thread d writes row d (16 values, 4
        // core-matrix chunks).
        auto stage_bv = [&]() {
            if (st_tid < D_H) {
                const uint4* src = reinterpret_cast<const uint4*>(a.BV + ((size_t)h * D_H + st_tid) * R);
                const uint4 w0 = src[0], w1 = src[1];
                const uint32_t wb[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                uint8_t* rowp = smem + OFF_BVF + (st_tid >> 3) * 512 + (st_tid & 7) * 16;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<float4*>(rowp + q4 * 128) = make_float4(
                        bf16lo(wb[2 * q4]), bf16hi(wb[2 * q4]), bf16lo(wb[2 * q4 + 1]), bf16hi(wb[2 * q4 + 1]));
            }
        };
        bool ok = true;
        if (!FUSED) {
            // Q~ row from TMEM -> bf16 -> shared memory (K-major, 32-byte swizzle), or with a
            // positional key back into TMEM as bf16 pairs (the A operand of its MMA).
            ok = wait_all(B(qt_mma), 0, a.status);
            tc_fence_after();
            // B^K has been consumed (qt_mma): without a positional key B_h^V takes its place.
            if (!ROPE) stage_bv();
            uint32_t v[16];
            tmem_ld_32x32b_x16(tmem + tl + TM_QT, v);
            uint32_t c[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) c[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
            if (ROPE) {
                tmem_st_32x32b_x8(tmem + tl + TM_QTB, c);
                tmem_wait_st();
            } else {
                const int sw = (row >> 2) & 1;
                *reinterpret_cast<uint4*>(smem + OFF_QT + row * 32 + ((0 ^ sw) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
                *reinterpret_cast<uint4*>(smem + OFF_QT + row * 32 + ((1 ^ sw) << 4)) = make_uint4(c[4], c[5], c[6], c[7]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(B(qt_ready));
        }

        const int qpos = qs + min(q0 + row, Tq - 1);
        float mref = -INFINITY, l = 0.f;
        for (int j = 0; j < nt; ++j) {
            if (!ok || aborted()) {
                ok = false;
                break;
            }
            ok = wait_all(B(s_full + (j & 1)), (j >> 1) & 1, a.status);
            if (!ok) break;
            tc_fence_after();
            // The whole S row comes out of TMEM in four back-to-back loads and one wait
            // (serial load -> wait round trips would dominate the tile), and stays in
            // registers for both passes: the row max (unscaled -- order-preserving under
            // the positive scale), then p = 2^(s * scale log2 e - m).
            const uint32_t sb = tmem + tl + ((j & 1) ? TM_S1 : TM_S0);
            const int k0 = j * kBN;
            const bool diag = k0 + kBN - 1 > qpos;
            uint32_t sv[kBN];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32_nowait(sb + c * 32, sv + c * 32);
            tmem_wait_ld();
            // Causal mask on diagonal tiles only: masked scores become -inf in the register
            // row, so the max and the exponentials below run without per-element branches
            // (2^-inf = 0).
            if (diag) {
                const int lim = qpos - k0;  // keys k0 + e with e <= lim are visible
#pragma unroll
                for (int e = 0; e < kBN; ++e) sv[e] = e <= lim ? sv[e] : 0xff800000u;
            }
            // eight independent partial maxima (one serial chain of 128 would stall on latency)
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = fmaxf(__uint_as_float(sv[i]), __uint_as_float(sv[8 + i]));
#pragma unroll
            for (int e = 16; e < kBN; e += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], __uint_as_float(sv[e + i]), __uint_as_float(sv[e + 8 + i]));
            float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
            mx *= a.scale_log2;
            const float mnew = fmaxf(mref, mx);
            const bool raise = mnew > mref + kRescaleThreshold;  // also true the first time a row sees a key
            const float muse = raise ? mnew : mref;
            const float alpha = raise ? ((mref == -INFINITY) ? 0.f : ex2_approx(mref - mnew)) : 1.f;
            // Key rows past the context may hold any bits: clear them before P . V reads them.
            const uint32_t kvb = OFF_V + (j % kVStages) * V_BYTES;
            if (k0 + kBN > ctx) {
                ok = wait_all(B(v_full + (j & 1)), (j >> 1) & 1, a.status);
                if (!ok) break;
                if (k0 + row >= ctx) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    uint4* rz = reinterpret_cast<uint4*>(smem + kvb + V_Z + row * 32);
#pragma unroll
                    for (int bk = 0; bk < NBV; ++bk) {
                        uint4* r0 = reinterpret_cast<uint4*>(smem + kvb + bk * 16384 + row * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) r0[i] = z;
                    }
                    rz[0] = z;
                    rz[1] = z;
                }
            }
            // p = 2^(s * scale log2 e - m) (one FFMA + one EX2), row sum, and the bf16 P row
            // back into TMEM over the first 64 columns of S_j (keys 2c, 2c+1 in column c),
            // where P_j . V_j takes its A operand from.
            float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            // A row that has seen no visible key yet (muse = -inf) gets p = 0 everywhere.
            const float nm = muse == -INFINITY ? -INFINITY : -muse;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t* v = sv + c * 32;
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(v[e]), a.scale_log2, nm));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(v[e + 1]), a.scale_log2, nm));
                    r8[(e >> 1) & 7] += p0 + p1;
                    pk[e / 2] = pack_bf16x2(p0, p1);
                }
                tmem_st_32x32b_x16(sb + c * 16, pk);
            }
            const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
            l = l * alpha + rs;
            mref = muse;
            // O may only be rescaled once P_{j-1} . V_{j-1} has finished accumulating into it;
            // without a rescale, P_j . V_j simply queues behind it in the tensor pipe.
            if (j > 0 && __any_sync(0xffffffffu, raise)) {
                ok = wait_all(B(o_done + ((j - 1) & 1)), ((j - 1) >> 1) & 1, a.status);
                if (!ok) break;
                tc_fence_after();
                uint32_t v[32];
#pragma unroll 1
                for (int c = 0; c < D_H / 32; ++c) {
                    tmem_ld_32x32b_x32(tmem + tl + TM_OS + c * 32, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st_32x32b_x32(tmem + tl + TM_OS + c * 32, v);
                }
                tmem_ld_32x32b_x16(tmem + tl + TM_OZ, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                tmem_st_32x32b_x16(tmem + tl + TM_OZ, v);
            }
            tmem_wait_st();
            fence_proxy_async_smem();  // zeroed value rows (if any) before the tensor core reads them
            tc_fence_before();
            mbar_arrive(B(p_full));
        }
        if (ROPE) {
            // Every S MMA has completed (S_{nt-1} was read above), so key stage 0 is free:
            // B_h^V goes there for the final MMA.  Arrive even on failure, so that MMA's wait ends.
            if (ok) stage_bv();
            fence_proxy_async_smem();
            mbar_arrive(B(bvf_ready));
        }
        // ---- epilogue: out = O_s / l (O_s already holds the B_h^V O_z term); absorbed weights:
        // out = [O_s | O_z] / l
        if (ok) ok = wait_all(B(fin_done), 0, a.status);
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int qrow = q0 + row;
#pragma unroll 1
            for (int c = 0; c < D_H / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + tl + TM_OS + c * 32, v);
                if (qrow < Tq) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        pk[e / 2] = pack_bf16x2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(out_row(qrow) + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            if (FUSED) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + tl + TM_OZ, v);
                if (qrow < Tq) {
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2)
                        pk[e / 2] = pack_bf16x2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(out_row(qrow) + D_H);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
        }
        if (!ok) *abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

template <int D_H, int D_R, bool FUSED>
static cudaError_t launch_prefill_tc_t(const PrefillMaps& maps, const PrefillArgs& a, cudaStream_t stream) {
    constexpr uint32_t smem = PfLayout<D_H, D_R>::SMEM;
    auto kern = prefill_tc_kernel<D_H, D_R, FUSED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.Tq + kBM - 1) / kBM, a.H, a.B);
    kern<<<grid, kThreads, smem, stream>>>(maps, a);
    return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const PrefillMaps& maps, const PrefillArgs& a, int d_h, int d_rope, cudaStream_t stream) {
    if (d_rope == 64) return d_h == 128 && !a.qt ? launch_prefill_tc_t<128, 64, false>(maps, a, stream) : cudaErrorInvalidValue;
    if (a.qt) return d_h == 64 ? launch_prefill_tc_t<64, 0, true>(maps, a, stream) : launch_prefill_tc_t<128, 0, true>(maps, a, stream);
    return d_h == 64 ? launch_prefill_tc_t<64, 0, false>(maps, a, stream) : launch_prefill_tc_t<128, 0, false>(maps, a, stream);
}

}  // namespace lrkv
