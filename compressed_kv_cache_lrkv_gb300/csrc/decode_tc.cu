// decode_tc.cu -- the split-K scan of the factored decode on the 5th-generation tensor cores,
// for 128 heads of d_h = 128 (the heads of a sequence are the M = 128 rows of the MMAs).
//
// Per sequence b, head h (Eqs. (6)-(7) of "Low-Rank Key Value Attention"; frames "Compute
// logits without expanding historical keys" and "Aggregate values before the residual
// up-projection"):  score_t = (q_h . s^K_t + q~_h . z^K_{h,t}) * scale,
//                   out_h   = sum_t p_t s^V_t + B_h^V (sum_t p_t z^V_{h,t}).
// The shared parts are products of the 128 x 128 query matrix Q (heads x features) with the
// shared key and value rows, one 8-token granule at a time:
//   S   = Q . [s^K_t]^T        tcgen05.mma M = 128, N = 16, K = 128 (kind::f16, fp32 in TMEM)
//   O  += P . [s^V_t]          tcgen05.mma M = 128, N = 128, K = 16
// Q and P are the A operands, read from TMEM.  A granule has 8 tokens but both MMAs work on
// 16: the descriptors' stride between 8-row groups points the second group at a 2 KB block of
// zeros after the ring, so tokens 8-15 are zero rows of s^K / s^V (and P's columns for them are
// zero).  The per-head latent products q~_h . z^K and p . z^V (each z element used once) run
// on the CUDA cores, two threads per head (four tokens of a granule each).
//
// Warp roles (320 threads): warp 0 streams the stages (the same four copies per granule as the
// CUDA-core scan: s^K and s^V by TMA tensor copies, z^K and z^V by bulk copies) into a ring;
// warp 1 allocates TMEM and issues the MMAs from one elected lane; warps 2-9 are the softmax,
// thread (warp, lane) owning head 32 (warp % 4) + lane = TMEM lane (a warp reaches only its
// lane quarter) and token half (warp - 2) / 4.  With one thread per head the latent products
// of a stage took four warps ~1.6 us and held the ring; two halve that.  The work plan, the pieces of work and the workspace partials are those of
// the CUDA-core scan (decode_work.cuh), so the absorb and combine kernels are shared.
//
// TMEM columns: Q 0-63 (bf16 pairs), S 64-79 / 80-95 (two buffers), P 96-103 / 104-111 (two
// buffers, bf16 pairs, columns 4-7 of each kept zero), O 128-255.
// The running maximum used for P is raised only when a row's maximum grows by more than 2^8
// (log2 units), so O is rarely rescaled in TMEM.
#include "decode_work.cuh"
#include "kernels.h"
#include "lrkv_internal.cuh"

namespace lrkv {

namespace {

constexpr int kTcThreads = 320;  // producer, MMA issuer, 8 softmax warps
constexpr uint32_t TC_Q = 0, TC_S = 64, TC_P = 96, TC_O = 128, TC_COLS = 256;
constexpr int kZeroBytes = 2048;  // two 64-column parts of 8 zero rows
constexpr float kTcRescale = 8.0f;

__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start / wait for the
// previous one's results (no-ops without the launch attribute).
__device__ __forceinline__ void pdl_trigger_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, const DecodeArgs& a) {
    const bool ok = mbar_wait_for(bar, parity, a.status, a.wait_ns);
    return __all_sync(0xffffffffu, ok);
}

}  // namespace

template <int R>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_split_tc_kernel(const __grid_constant__ CUtensorMap tm_sK, const __grid_constant__ CUtensorMap tm_sV,
                           const DecodeArgs a) {
    constexpr int D_H = 128, D_K = 128, H = 128, W = D_H + R, NC = R / 8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t smem_s = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nslot = a.nslot, stage_bytes = a.stage_bytes;

    // [ring][zero block][barriers][meta][lengths][pair exchange][plan][TMEM address, abort flag]
    uint8_t* zero = smem + nslot * stage_bytes;  // 1024-aligned (stage_bytes is a multiple of 1024)
    const uint32_t Z = smem_u32(zero);
    uint64_t* bars = reinterpret_cast<uint64_t*>(zero + kZeroBytes);
    uint64_t* full = bars;                  // [nslot] a stage landed
    uint64_t* empty = bars + nslot;         // [nslot] softmax warps (8) and the MMAs (1) are done with it
    uint64_t* s_full = bars + 2 * nslot;    // [2] S_j in TMEM buffer j % 2
    uint64_t* p_full = s_full + 2;          // [2] P_j written (4 warps)
    uint64_t* o_done = p_full + 2;          // [2] O += P_j . V_j complete
    uint64_t* q_ready = o_done + 2;         // Q of the segment in TMEM (4 warps)
    uint64_t* o_free = q_ready + 1;         // O of the segment read out (4 warps)
    uint64_t* drain = o_free + 1;           // every MMA of the CTA complete
    int* meta = reinterpret_cast<int*>(drain + 1);  // [nslot] 1: stage holds data
    int* slc = meta + ((nslot + 3) & ~3);           // first kSeqCache sequence lengths
    float* xbuf = reinterpret_cast<float*>(slc + kSeqCache);  // [2][H][8] latent logits, then [H][R] accumulators
    Work* plan = reinterpret_cast<Work*>(xbuf + 2 * 128 * kGran + 128 * R);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(plan + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto aborted = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0); };

    if (threadIdx.x == 0) {
        prefetch_tmap(&tm_sK);
        prefetch_tmap(&tm_sV);
        for (int s = 0; s < nslot; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 9);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&p_full[i]), 4);
            mbar_init(smem_u32(&o_done[i]), 1);
        }
        mbar_init(smem_u32(q_ready), 4);
        mbar_init(smem_u32(o_free), 4);
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kZeroBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(zero)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int b = threadIdx.x; b < a.B && b < kSeqCache; b += blockDim.x) slc[b] = a.seq_lens[b];
    fence_proxy_async_smem();  // the zero block is read by the tensor cores
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TC_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        Work w{a.seq_lens, slc, a.B, a.layers, a.max_pages * kBlockSize, a.nranges, 0, 0, 1, 0};
        w.lgh = 0;
        w.plan<32>(a.bubble, lane);
        if (lane == 0) *plan = w;
    }
    __syncthreads();
    const Work wk = *plan;
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        SegWalk walk;
        walk.start(blockIdx.x);
        int vb = 0, sg0 = 0, sg1 = 0, pslot = 0;
        int g = 0;  // stages issued so far (ring position and phase)
        bool ok = true;
        while (ok && walk.next(wk, &vb, &sg0, &sg1, &pslot)) {
            const int l = vb / a.B, bb = vb - l * a.B;
            const int pg0 = sg0 >> 3;
            const int32_t* bt_row = a.block_table + (size_t)bb * a.max_pages;
            int batch = -1, pid = -1;
            for (int gi = sg0; gi < sg1; ++gi, ++g) {
                const int pi = (gi >> 3) - pg0;  // page of the segment; lane i holds page 32 batch + i
                if ((pi >> 5) != batch) {
                    batch = pi >> 5;
                    const int pp = pg0 + batch * 32 + lane;
                    pid = pp < a.max_pages ? bt_row[pp] : -1;
                }
                const int blk = __shfl_sync(0xffffffffu, pid, pi & 31);
                const int s = g % nslot;
                if (g >= nslot && !tc_wait(smem_u32(&empty[s]), ((g / nslot) - 1) & 1, a)) {
                    ok = false;
                    break;
                }
                if (aborted()) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t st = smem_s + s * stage_bytes, bar = smem_u32(&full[s]);
                    if (blk < 0 || blk >= a.num_blocks) {
                        set_status(a.status, LRKV_DEV_BAD_BLOCK);
                        meta[s] = 0;
                        mbar_arrive(bar);
                    } else {
                        meta[s] = 1;
                        mbar_arrive_expect_tx(bar, 16u * (D_K + D_H) + 32u * H * R);
                        const int row = blk * kBlockSize + ((gi & 7) << 3);
                        tma_load_4d_hint(st, &tm_sK, 0, row, 0, l, bar, pol);
                        tma_load_4d_hint(st + 16 * D_K, &tm_sV, 0, row, 0, l, bar, pol);
                        const size_t zoff = (size_t)row * H * R;
                        bulk_load_hint(st + 16 * (D_K + D_H), a.zK + l * a.ls_zK + zoff, 16u * H * R, bar, pol);
                        bulk_load_hint(st + 16 * (D_K + D_H) + 16 * H * R, a.zV + l * a.ls_zV + zoff, 16u * H * R,
                                       bar, pol);
                    }
                }
                __syncwarp();
            }
        }
        if (!ok) {
            *abort_flag = 1;
            // let the copies still in flight land before the CTA exits (always the full limit)
            if (lane == 0)
                for (int k = max(0, g - nslot); k < g; ++k) mbar_wait(smem_u32(&full[k % nslot]), (k / nslot) & 1, a.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        constexpr uint32_t id_S = idesc_bf16_f32(128, 16);
        constexpr uint32_t id_PV = idesc_bf16_f32(128, 128) | (1u << 16);  // B (s^V) MN-major
        SegWalk walk;
        walk.start(blockIdx.x);
        int vb = 0, sg0 = 0, sg1 = 0, pslot = 0;
        int g = 0, segn = 0;
        bool ok = true;
        while (ok && walk.next(wk, &vb, &sg0, &sg1, &pslot)) {
            const int nst = sg1 - sg0;
            ok = !aborted() && tc_wait(smem_u32(q_ready), segn & 1, a);  // this segment's Q in TMEM
            for (int k = 0; ok && k <= nst; ++k) {
                if (k < nst) {
                    // S_k = Q . [s^K of the stage | 8 zero rows]^T into buffer (g + k) % 2.  That buffer's
                    // previous S was read before its P was written (p_full, waited below for the P.V).
                    const int gk = g + k, s = gk % nslot, b = gk & 1;
                    if (aborted() || !tc_wait(smem_u32(&full[s]), (gk / nslot) & 1, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sK = smem_s + s * stage_bytes;
                    const uint32_t dS = tmem + TC_S + 16 * b;
#pragma unroll
                    for (int kk = 0; kk < D_K / 16; ++kk) {
                        // K step kk: 64-column part kk / 4, 32 bytes into its rows; the second 8-row
                        // group (tokens 8-15) is the zero block, (Z - sK) bytes on
                        const uint64_t bd = sdesc(sK + (kk >> 2) * 1024 + (kk & 3) * 32, 16, Z - sK, 2);
                        if (elect_one_sync()) tc_mma_bf16_ts(dS, tmem + TC_Q + kk * 8, bd, id_S, kk > 0);
                    }
                    if (elect_one_sync()) tc_commit(smem_u32(&s_full[b]));
                    __syncwarp();
                }
                if (k >= 1) {
                    // O (+)= P_{k-1} . [s^V of its stage ; 8 zero rows]
                    const int gp = g + k - 1, s = gp % nslot, b = gp & 1;
                    if (aborted() || !tc_wait(smem_u32(&p_full[b]), (gp >> 1) & 1, a) ||
                        (k == 1 && segn > 0 && !tc_wait(smem_u32(o_free), (segn - 1) & 1, a))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sV = smem_s + s * stage_bytes + 16 * D_K;
                    const uint64_t bd = sdesc(sV, 1024, Z - sV, 2);  // parts 1 KB apart; tokens 8-15: zero block
                    if (elect_one_sync()) {
                        tc_mma_bf16_ts(tmem + TC_O, tmem + TC_P + 8 * b, bd, id_PV, k > 1);
                        tc_commit(smem_u32(&o_done[b]));
                        tc_commit(smem_u32(&empty[s]));
                    }
                    __syncwarp();
                }
            }
            g += nst;
            ++segn;
        }
        if (!ok) *abort_flag = 1;
        // every MMA this warp issued has finished before TMEM is released
        if (elect_one_sync()) tc_commit(smem_u32(drain));
        __syncwarp();
        tc_wait(smem_u32(drain), 0, a);
    } else {
        // ------------------------------------------------------------------ softmax: two threads per head
        // Warps 2-9: quarter q = warp % 4 of the TMEM lanes (head 32 q + lane), token half th = 0
        // (warps 2-5) or 1 (warps 6-9) of every granule.  Each thread forms the latent logits and
        // accumulates the latent values of its four tokens; the pair exchanges the logits through
        // shared memory (a named barrier per quarter), both run the same softmax on all eight, and
        // the th = 0 thread alone writes P, rescales O and writes the partial.
        const int q4 = warp & 3, th = (warp - 2) >> 2;
        const int h = q4 * 32 + lane;  // = this thread's TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);  // the warp's lane quarter
        const int pair_bar = 1 + q4;                              // named barrier of the two warps of the quarter
        auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
        // Every thread of a pair passes the same pair barriers: it walks all its segments and stages
        // whatever happens; after an expired wait (or another role's abort) `bad` skips the waits and
        // the work, never the barriers.
        SegWalk walk;
        walk.start(blockIdx.x);
        int vb = 0, sg0 = 0, sg1 = 0, pslot = 0;
        int g = 0, segn = 0;
        bool bad = false;
        bool qt_ready = false;
        auto check = [&](bool waited) {  // a failed wait: stop waiting, flag the abort
            if (!waited) {
                bad = true;
                *abort_flag = 1;
            }
        };
        if (th == 0) {  // P columns 4-7 (tokens 8-15) of both buffers stay zero
            const uint32_t z8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            tmem_st_x8(tl + TC_P, z8);
            tmem_st_x8(tl + TC_P + 8, z8);
            tmem_wait_st();
        }
        while (walk.next(wk, &vb, &sg0, &sg1, &pslot)) {
            const int l = vb / a.B, bb = vb - l * a.B;
            const int L = bb < kSeqCache ? slc[bb] : a.seq_lens[bb];
            const int nst = sg1 - sg0;
            if (aborted()) bad = true;
            if (warp == 2 && lane == 0 && sg0 == 0) {
                // a sequence's first segment records where its partials are, for the combine
                const int gr = wk.gran(vb);
                const int np = wk.pieces ? wk.npieces(vb % wk.B, wk.chunk)
                                         : wk.range_of(walk.seg_start + gr - 1) - (pslot - vb) + 1;
                a.seg_table[vb] = make_int2(pslot, np);
            }
            if (!qt_ready) {
                pdl_wait_grid();  // q~ written by the absorb kernel (no-op for an ordinary launch)
                qt_ready = true;
            }
            float qt[R];
            if (a.qt_in) {  // absorbed query weights: q~ in bf16 from the caller
                const uint4* qr = reinterpret_cast<const uint4*>(a.qt_in + l * a.ls_qt + ((size_t)bb * H + h) * R);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const uint4 x = qr[c];
                    qt[8 * c + 0] = bf16lo(x.x);
                    qt[8 * c + 1] = bf16hi(x.x);
                    qt[8 * c + 2] = bf16lo(x.y);
                    qt[8 * c + 3] = bf16hi(x.y);
                    qt[8 * c + 4] = bf16lo(x.z);
                    qt[8 * c + 5] = bf16hi(x.z);
                    qt[8 * c + 6] = bf16lo(x.w);
                    qt[8 * c + 7] = bf16hi(x.w);
                }
            } else {  // q~ = q B^K from the absorb kernel, fp32
                const float4* qr = reinterpret_cast<const float4*>(a.qt + ((size_t)vb * H + h) * R);
#pragma unroll
                for (int c = 0; c < R / 4; ++c) {
                    const float4 x = qr[c];
                    qt[4 * c] = x.x;
                    qt[4 * c + 1] = x.y;
                    qt[4 * c + 2] = x.z;
                    qt[4 * c + 3] = x.w;
                }
            }
            if (th == 0 && !bad) {
                // the query row q_h into TMEM (Q, the A operand of S); the previous segment's Q is no
                // longer read (its last S was waited for)
                const uint4* qrow = reinterpret_cast<const uint4*>(a.q + l * a.ls_q + ((size_t)bb * H + h) * D_K);
                uint32_t qv[32];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 x = qrow[half * 8 + c];
                        qv[4 * c] = x.x;
                        qv[4 * c + 1] = x.y;
                        qv[4 * c + 2] = x.z;
                        qv[4 * c + 3] = x.w;
                    }
                    tmem_st_32x32b_x32(tl + TC_Q + 32 * half, qv);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(q_ready));
            }
            float mref = -INFINITY, lsum = 0.f;
            float accz[R];
#pragma unroll
            for (int i = 0; i < R; ++i) accz[i] = 0.f;
            bool o_started = false;
            for (int k = 0; k < nst; ++k) {
                const int gk = g + k, s = gk % nslot, b = gk & 1;
                if (!bad && aborted()) bad = true;
                if (!bad) check(tc_wait(smem_u32(&full[s]), (gk / nslot) & 1, a));
                const int t0 = (sg0 + k) * kGran;
                const int nvalid = (!bad && meta[s]) ? min(kGran, L - t0) : 0;
                const uint8_t* st = smem + s * stage_bytes;
                const uint8_t* zK = st + 16 * (D_K + D_H);
                const uint8_t* zV = zK + 16 * H * R;
                // latent logits q~_h . z^K_{h,t} of this thread's four tokens (CUDA cores), to the pair
                float* xs = xbuf + (b * H + h) * kGran;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = 4 * th + i;
                    float acc = 0.f;
                    if (t < nvalid) {
                        const uint4* row = reinterpret_cast<const uint4*>(zK + ((size_t)t * H + h) * R * 2);
#pragma unroll
                        for (int cc = 0; cc < NC; ++cc) {
                            const uint4 v = row[cc];
                            acc = fmaf(qt[cc * 8 + 0], bf16lo(v.x), acc);
                            acc = fmaf(qt[cc * 8 + 1], bf16hi(v.x), acc);
                            acc = fmaf(qt[cc * 8 + 2], bf16lo(v.y), acc);
                            acc = fmaf(qt[cc * 8 + 3], bf16hi(v.y), acc);
                            acc = fmaf(qt[cc * 8 + 4], bf16lo(v.z), acc);
                            acc = fmaf(qt[cc * 8 + 5], bf16hi(v.z), acc);
                            acc = fmaf(qt[cc * 8 + 6], bf16lo(v.w), acc);
                            acc = fmaf(qt[cc * 8 + 7], bf16hi(v.w), acc);
                        }
                    }
                    xs[t] = acc;
                }
                // Masked tokens' s^V rows are zeroed: P is 0 there, and 0 times stale bits could be NaN.
                if (th == 0 && !bad && nvalid < kGran) {
                    for (int i = threadIdx.x - 64; i < 2 * kGran * 8; i += 128) {
                        const int part = i >> 6, t = (i >> 3) & 7, ch = i & 7;
                        if (t >= nvalid)
                            reinterpret_cast<uint4*>(smem + s * stage_bytes + 16 * D_K + part * 1024 + t * 128)[ch] =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                // S_k from TMEM
                if (!bad) check(tc_wait(smem_u32(&s_full[b]), (gk >> 1) & 1, a));
                float sv[kGran];
                if (!bad) {
                    tc_fence_after();
                    tmem_ld_x8(tl + TC_S + 16 * b, sv);
                }
                pair_sync();  // the partner's latent logits are in xs
                float mx = -INFINITY;
#pragma unroll
                for (int t = 0; t < kGran; ++t) {
                    sv[t] = t < nvalid ? (sv[t] + xs[t]) * a.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sv[t]);
                }
                // Raise the reference maximum only when it is exceeded by more than 2^8; O, l and
                // the latent accumulators are rescaled then (O in TMEM, after every issued P.V).
                const bool raise = mx > mref + kTcRescale || (mref == -INFINITY && mx != -INFINITY);
                if (__any_sync(0xffffffffu, raise)) {
                    const float nref = raise ? mx : mref;
                    const float alpha = (mref == -INFINITY) ? 0.f : exp2f(mref - nref);
                    lsum *= alpha;
#pragma unroll
                    for (int i = 0; i < R; ++i) accz[i] *= alpha;
                    if (th == 0 && o_started && !bad) check(tc_wait(smem_u32(&o_done[(gk - 1) & 1]), ((gk - 1) >> 1) & 1, a));
                    if (th == 0 && o_started && !bad) {
                        tc_fence_after();
                        const float sc = raise ? alpha : 1.f;
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            uint32_t ov[32];
                            tmem_ld_32x32b_x32(tl + TC_O + 32 * c, ov);
#pragma unroll
                            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * sc);
                            tmem_st_32x32b_x32(tl + TC_O + 32 * c, ov);
                        }
                        tmem_wait_st();
                    }
                    mref = nref;
                }
                float p[kGran];
#pragma unroll
                for (int t = 0; t < kGran; ++t) {
                    p[t] = (t < nvalid) ? exp2f(sv[t] - mref) : 0.f;
                    lsum += p[t];
                }
                if (th == 0 && gk >= 2 && !bad) check(tc_wait(smem_u32(&o_done[b]), ((gk - 2) >> 1) & 1, a));
                if (th == 0 && !bad) {
                    // P_k into buffer b, once the P.V two stages back (its previous content) is done
                    const uint32_t pw[8] = {pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                                            pack_bf16x2(p[6], p[7]), 0u, 0u, 0u, 0u};
                    tmem_st_x8(tl + TC_P + 8 * b, pw);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&p_full[b]));
                }
                o_started = true;
                // latent values p . z^V_{h,t} of this thread's four tokens (CUDA cores)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = 4 * th + i;
                    if (t < nvalid) {
                        const uint4* row = reinterpret_cast<const uint4*>(zV + ((size_t)t * H + h) * R * 2);
#pragma unroll
                        for (int cc = 0; cc < NC; ++cc) {
                            const uint4 v = row[cc];
                            accz[cc * 8 + 0] = fmaf(p[t], bf16lo(v.x), accz[cc * 8 + 0]);
                            accz[cc * 8 + 1] = fmaf(p[t], bf16hi(v.x), accz[cc * 8 + 1]);
                            accz[cc * 8 + 2] = fmaf(p[t], bf16lo(v.y), accz[cc * 8 + 2]);
                            accz[cc * 8 + 3] = fmaf(p[t], bf16hi(v.y), accz[cc * 8 + 3]);
                            accz[cc * 8 + 4] = fmaf(p[t], bf16lo(v.z), accz[cc * 8 + 4]);
                            accz[cc * 8 + 5] = fmaf(p[t], bf16hi(v.z), accz[cc * 8 + 5]);
                            accz[cc * 8 + 6] = fmaf(p[t], bf16lo(v.w), accz[cc * 8 + 6]);
                            accz[cc * 8 + 7] = fmaf(p[t], bf16hi(v.w), accz[cc * 8 + 7]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0 && !bad) mbar_arrive(smem_u32(&empty[s]));  // this warp is done with the stage's latents
            }
            // The segment's partial: (m, l), O (from TMEM, after its last P.V) and the sum of the
            // pair's latent accumulators, into the workspace row [head][slot].
            float* ax = xbuf + 2 * H * kGran + h * R;  // the th = 1 half of the latent accumulator
            if (th == 1) {
#pragma unroll
                for (int i = 0; i < R; ++i) ax[i] = accz[i];
            }
            pair_sync();
            if (th == 0 && !bad) check(tc_wait(smem_u32(&o_done[(g + nst - 1) & 1]), ((g + nst - 1) >> 1) & 1, a));
            if (th == 0 && !bad) {
                tc_fence_after();
                float* pacc = a.part_acc + ((size_t)h * a.pmax + pslot) * W;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t ov[32];
                    tmem_ld_32x32b_x32(tl + TC_O + 32 * c, ov);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        reinterpret_cast<float4*>(pacc + 32 * c)[i] =
                            make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                                        __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
                }
#pragma unroll
                for (int i = 0; i < R / 4; ++i)
                    reinterpret_cast<float4*>(pacc + D_H)[i] =
                        make_float4(accz[4 * i] + ax[4 * i], accz[4 * i + 1] + ax[4 * i + 1],
                                    accz[4 * i + 2] + ax[4 * i + 2], accz[4 * i + 3] + ax[4 * i + 3]);
                *reinterpret_cast<float2*>(a.part_ml + ((size_t)h * a.pmax + pslot) * 2) = make_float2(mref, lsum);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(o_free));
            }
            pair_sync();  // the exchange area is free again
            g += nst;
            ++segn;
        }
    }
    pdl_trigger_grid();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TC_COLS);
}

int decode_tc_smem_bytes(int nslot, int stage_bytes) {
    // ring, zero block, barriers (2 nslot + 9), meta, lengths, pair exchange (for r <= 16), plan,
    // TMEM address + abort flag, alignment
    return nslot * stage_bytes + kZeroBytes + (2 * nslot + 9) * 8 + ((nslot + 3) & ~3) * 4 + kSeqCache * 4 +
           (2 * 128 * kGran + 128 * 16) * 4 + (int)sizeof(Work) + 16 + 1024;
}

template <int R>
cudaError_t launch_decode_tc_split(const CUtensorMap& tK, const CUtensorMap& tV, const DecodeArgs& a, int grid,
                                   int smem_bytes, bool pdl, cudaStream_t stream) {
    auto k = decode_split_tc_kernel<R>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, tK, tV, a);
}

template cudaError_t launch_decode_tc_split<8>(const CUtensorMap&, const CUtensorMap&, const DecodeArgs&, int, int,
                                               bool, cudaStream_t);
template cudaError_t launch_decode_tc_split<16>(const CUtensorMap&, const CUtensorMap&, const DecodeArgs&, int, int,
                                                bool, cudaStream_t);

}  // namespace lrkv
