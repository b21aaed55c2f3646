// decode.cu -- factored LRKV decode (Eqs. (6)-(7) of "Low-Rank Key Value Attention").
//
// Per sequence b and head h, with q~_h = q_h B_h^K (frame "Compute logits without
// expanding historical keys", step 1):
//     score_t = (q_h . s^K_t + q~_h . z^K_{h,t}) * scale
//     out_h   = sum_t p_t s^V_t + B_h^V (sum_t p_t z^V_{h,t})       (Eq. (7))
// Per-head K_h / V_h are never formed.
// With a decoupled positional key (D_R > 0) the shared key row is [s^K | k^R] and the
// query [q | q^R]: the tensor-core logits simply run over D_K = D_H + D_R columns,
// while q~ = q B^K uses the first D_H of them.
//
// One call may cover several layers (each with its own cache pools, q, B^K, B^V and
// output, found at per-layer strides, all sharing the block table and lengths): every
// (layer, sequence) pair is a "virtual sequence", and one launch of each kernel serves them all.
//
// Kernel 0 (absorb): q~ for every (virtual sequence, head) into the workspace, fp32.
// Kernel 1 (split): a persistent grid of at most one CTA per SM, launched with
//   programmatic dependent launch so it starts streaming while kernel 0 runs.
//   The cached tokens of all virtual sequences are cut into 8-token granules; the
//   granules, concatenated, are divided into equal contiguous ranges (one per SM
//   unless the caller sets the count), each covering pieces ("segments") of one or
//   more consecutive sequences.  Each granule's s^K, s^V (TMA tensor loads, 128-byte
//   swizzle) and z^K, z^V (bulk copies) go into a ring of shared-memory stages, read
//   from HBM once for all H heads.  Consumer warps own 16 heads each; NG groups of
//   ceil(H/16) warps take stages round-robin with their own online-softmax state,
//   merged inside the CTA at the end of each segment into one partial
//   (m, l, acc_s[d_h], acc_z[r]) per head.
//     - q . s^K and p . s^V run on the tensor cores (mma.sync m16n8k16 / m16n8k8,
//       heads on M, tokens on N / K) -- s is shared by all heads of the CTA;
//     - q~ . z^K and p . z^V run on CUDA cores in fp32 (each z element is used
//       once; nothing for a tensor core to reuse).
// Kernel 2 (combine): log-sum-exp merge of each (sequence, head)'s partials, the residual
//   up-projection B_h^V acc_z, the bf16 store (also a dependent launch).
#include "decode_work.cuh"
#include "kernels.h"
#include "lrkv_internal.cuh"

namespace lrkv {

// Cooperative copy of the first kSeqCache lengths (caller synchronises afterwards).
__device__ __forceinline__ void stage_seq_lens(int* dst, const int32_t* src, int B, int tid, int nthreads) {
    for (int b = tid; b < B && b < kSeqCache; b += nthreads) dst[b] = src[b];
}

// Index of (head row h, token t) in a warp's 16 x 8 scratch of z-scores or probabilities.  The
// token index is XOR-ed with bits 2-3 of h, so that both the stores and loads by (head, four
// tokens) lanes and those by the (row group, token pair) lanes of the MMA fragments hit 32
// different banks.
__device__ __forceinline__ int sidx(int h, int t) { return h * 8 + (t ^ ((h >> 2) & 3)); }

// Bounded wait until a slot's stage tag equals `want` (sets LRKV_DEV_TIMEOUT on expiry).
__device__ __forceinline__ bool wait_tag(volatile int* tag, int want, uint32_t* status, uint64_t limit_ns) {
    if (*tag == want) return true;
    const uint64_t t0 = globaltimer_ns();
    while (*tag != want) {
        __nanosleep(32);
        if (globaltimer_ns() - t0 > limit_ns) {
            set_status(status, LRKV_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void named_bar(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start, and
// wait for the previous one's results (both no-ops without the launch attribute).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ kernel 0
// q~[vb][h][j] = sum_d q[vb][h][d] B^K[h][d][j]; one block per (head, virtual sequence):
// 256 / R slices of the d range are summed in parallel, then reduced in
// shared memory, so all of B_h^K (d_h x r) is in flight at once.
// Launched as a dependent of the caller's previous kernel on the stream, so its blocks are in
// place when that kernel ends; it waits for that kernel's completion before touching memory and
// only then lets the scan start (the scan reads the cache, which the previous kernel -- an
// append of the newest rows -- may have written).
template <int D_H, int R, int D_R>
__global__ void __launch_bounds__(256) decode_absorb_kernel(const DecodeArgs a) {
    pdl_wait();
    pdl_trigger();
    constexpr int NS = 256 / R;           // d slices
    constexpr int DS = D_H / NS;          // d values per slice (>= 2)
    static_assert(DS >= 1 && D_H % NS == 0, "slices");
    const int h = blockIdx.x, vb = blockIdx.y;
    const int l = vb / a.B, b = vb - l * a.B;
    const int j = threadIdx.x % R, sl = threadIdx.x / R;
    __shared__ float part[NS][R];
    const uint16_t* qrow = a.q + l * a.ls_q + ((size_t)b * a.H + h) * (D_H + D_R) + sl * DS;
    const uint16_t* bk = a.BK + l * a.ls_BK + ((size_t)h * D_H + sl * DS) * R + j;
    float acc = 0.f;
#pragma unroll
    for (int dd = 0; dd < DS; ++dd)
        acc = fmaf(__uint_as_float((uint32_t)qrow[dd] << 16), __uint_as_float((uint32_t)bk[dd * R] << 16), acc);
    part[sl][j] = acc;
    __syncthreads();
    if (threadIdx.x < R) {
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < NS; ++i) v += part[i][threadIdx.x];
        a.qt[((size_t)vb * a.H + h) * R + threadIdx.x] = v;
    }
}

// Issue the loads of one stage -- GS 8-token granules from granule gi (GS-aligned, inside one
// page) -- of block `blk` of layer `l` into a ring slot:
// s^K (with k^R when D_R > 0) and s^V by one TMA tensor copy each (128-byte swizzle; the map
// views a row as 64-column parts 128 bytes apart, so one box brings all parts of the 8 rows),
// z^K, z^V by bulk copies.  An out-of-range block id is reported and the stage is marked empty.
// (One thread issues all four: spreading them over four lanes of the refilling warp made each
// refill cheaper but the H = 128 decode slower as a whole.)
// With head groups, z^K and z^V of the group's HL heads come by one tensor copy each (the 8
// tokens' slices of HL r elements, in 256-byte pieces, landing as [token][head][r]).
template <int D_H, int R, int D_R, bool HG, int GS>
__device__ __forceinline__ void issue_stage(const CUtensorMap* tm_sK, const CUtensorMap* tm_sV,
                                            const CUtensorMap* tm_zK, const CUtensorMap* tm_zV, const DecodeArgs& a,
                                            uint32_t st, uint32_t bar, int* meta_slot, int l, int blk, int gi,
                                            int hbase, int HL, uint64_t pol, uint64_t pol_s) {
    if (blk < 0 || blk >= a.num_blocks) {
        set_status(a.status, LRKV_DEV_BAD_BLOCK);
        *meta_slot = 0;
        mbar_arrive(bar);
        return;
    }
    *meta_slot = 1;
    constexpr int D_K = D_H + D_R;
    mbar_arrive_expect_tx(bar, GS * (16u * (D_K + D_H) + 32u * HL * R));
    const int row = blk * kBlockSize + ((gi & 7) << 3);
    // one copy per shared part: the 8 GS rows' 64-column parts land as [part][row][64], GS KB per part
    tma_load_4d_hint(st, tm_sK, 0, row, 0, l, bar, pol_s);
    tma_load_4d_hint(st + 16 * D_K * GS, tm_sV, 0, row, 0, l, bar, pol_s);
    const uint32_t zst = st + 16 * GS * (D_K + D_H);
    if (HG && a.nhg > 1) {  // (head groups come with one-granule stages)
        const int piece = hbase * R / 128;  // the group's first 128-element piece of a token's latents
        tma_load_4d_hint(zst, tm_zK, 0, piece, row, l, bar, pol);
        tma_load_4d_hint(zst + 16 * HL * R, tm_zV, 0, piece, row, l, bar, pol);
    } else {
        const size_t zoff = (size_t)row * a.H * R;
        bulk_load_hint(zst, a.zK + l * a.ls_zK + zoff, 16u * GS * a.H * R, bar, pol);
        bulk_load_hint(zst + 16 * GS * a.H * R, a.zV + l * a.ls_zV + zoff, 16u * GS * a.H * R, bar, pol);
    }
}

// ------------------------------------------------------------------ kernel 1
// At most 8 warps per CTA (one per head tile and group), so each thread may
// hold up to 255 registers.  There is no dedicated producer warp: thread 0
// fills the ring at the start of each segment, and afterwards the last warp to
// release a stage refills that slot with the stage nslot positions ahead.
template <int D_H, int R, int D_R, bool HG, int GS>
__global__ void __launch_bounds__(256, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_sK, const __grid_constant__ CUtensorMap tm_sV,
                        const __grid_constant__ CUtensorMap tm_zK, const __grid_constant__ CUtensorMap tm_zV,
                        const DecodeArgs a) {
    static_assert(D_H == 64 || D_H == 128, "d_h");
    static_assert(D_R == 0 || D_R == 64, "d_rope");
    static_assert(R % 8 == 0 && R <= 32, "r");
    constexpr int D_K = D_H + D_R;                              // shared key row [s^K | k^R]
    constexpr int NC = R / 8;                                   // 16-byte chunks per z row
    constexpr int RP128 = (2 * R >= 128) ? 1 : 128 / (2 * R);   // z rows per 128-byte bank line
    constexpr int W = D_H + R;                                  // accumulator width per head
    constexpr int WS = decode_stage_stride(W);                  // its row stride in the group staging

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t smem_s = smem_u32(smem);

    const int H = a.H;                                           // all heads (global layouts)
    // head groups (HG: compiled only where they can occur; without them the group terms fold away)
    const int nhg = HG ? a.nhg : 1;
    const int lgh = nhg == 8 ? 3 : nhg == 4 ? 2 : nhg == 2 ? 1 : 0;
    const int HL = H >> lgh;                                     // heads of one group: this CTA's share
    const int HT = (HL + 15) >> 4;
    const int NCW = HT * a.ng;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nslot = a.nslot;
    const int stage_bytes = a.stage_bytes;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + nslot * stage_bytes);
    int* meta = reinterpret_cast<int*>(full + nslot);            // 1: stage holds data, 0: skipped
    int* rel = meta + nslot;                                     // warps done with the slot's current stage
    int* nissued = rel + nslot;                                  // stages ever issued into the slot
    volatile int* tag = nissued + nslot;                         // CTA-wide index of the stage last issued
    int* pages = meta + ((4 * nslot + 3) & ~3);                  // block ids of the current split's pages
    int* slc = pages + kPageCache;                               // first kSeqCache sequence lengths
    float* scratch = reinterpret_cast<float*>(slc + kSeqCache);
    volatile int* abort_flag = reinterpret_cast<int*>(scratch + NCW * kScratchFloats);
    SplitCtl* ctl = reinterpret_cast<SplitCtl*>((reinterpret_cast<uintptr_t>(abort_flag) + 16) & ~(uintptr_t)15);

    if (threadIdx.x == 0) {
        prefetch_tmap(&tm_sK);
        prefetch_tmap(&tm_sV);
        if (nhg > 1) {
            prefetch_tmap(&tm_zK);
            prefetch_tmap(&tm_zV);
        }
        for (int s = 0; s < nslot; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            rel[s] = 0;
            nissued[s] = 0;
            tag[s] = -1;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    stage_seq_lens(slc, a.seq_lens, a.B, threadIdx.x, blockDim.x);
    // The block table is read right after the plan: start bringing it into L2.
    if ((size_t)a.B * a.max_pages <= kBtPrefetchEntries)
        for (int off = threadIdx.x * 32; off < a.B * a.max_pages; off += blockDim.x * 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.block_table + off));
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    // the shared rows are read by every head group's CTA: not evict-first then
    const uint64_t pol_s = nhg > 1 ? policy_evict_normal() : pol;
    // Warp 0 plans the work (lanes over the sequences) and steps to this CTA's first segment.
    if (warp == 0) {
        Work w{a.seq_lens, slc, a.B << lgh, a.layers, a.max_pages * kBlockSize, a.nranges, 0, 0, 1, 0};
        w.lgh = lgh;
        w.plan<32>(a.bubble, lane);
        if (lane == 0) {
            ctl->wk = w;
            ctl->walk.start(blockIdx.x);
            ctl->advance(a.seg_table);
        }
    }

    const int grp = warp / HT, ht = warp % HT;
    const int h0 = ht * 16;
    const int g = lane >> 2, tq = lane & 3;
    const int hz = lane & 15, half = lane >> 4;
    const int hzh = h0 + hz;
    const bool hz_ok = hzh < HL;
    const int rot = (hz / RP128) % NC;
    float* SZ = scratch + warp * kScratchFloats;
    float* SP = SZ + 128;
    float* SA = SP + 128;
    const int nct = NCW * 32;
    const int hA = h0 + g, hB = h0 + g + 8;
    bool qt_ready = false;

    int kbase = 0;  // stages consumed by this CTA before the current segment (ring position and phase)
    for (;;) {
        // Once every warp is here the previous segment is fully consumed and merged:
        // no copy is in flight and the ring memory is free.
        // (the descriptor of this segment was stepped to by thread 0 during the previous one)
        named_bar(1, nct);
        if (!ctl->valid) break;
        const int vb = ctl->vb, sg0 = ctl->g0, sg1 = ctl->g1, pslot = ctl->slot;
        const int vbr = vb >> lgh;                       // the (layer, sequence) pair
        const int hbase = (vb & (nhg - 1)) * HL;         // first head of this segment's group
        const int l = vbr / a.B, bb = vbr - (vbr / a.B) * a.B;
        const int L = bb < kSeqCache ? slc[bb] : a.seq_lens[bb];
        // stages: GS-granule blocks, aligned in the sequence, that meet [sg0, sg1)
        const int base0 = sg0 & ~(GS - 1);
        const int nst = GS == 1 ? sg1 - sg0 : (sg1 - 1) / GS - sg0 / GS + 1;
        const int pg0 = sg0 >> 3;
        const int32_t* bt_row = a.block_table + (size_t)bb * a.max_pages;

        for (int i = threadIdx.x; i < kPageCache && pg0 + i < a.max_pages; i += nct) pages[i] = bt_row[pg0 + i];
        fence_proxy_async_smem();  // generic accesses of the ring (merge) before async-proxy refills
        named_bar(1, nct);
        // Fill the ring.  A copy instruction costs its thread ~60-80 ns (~0.4 us a stage), so a
        // long fill (many small stages) is spread over the warps, stage k by warp k mod NCW;
        // a short one stays with thread 0, which measured faster there.
        const int nfill = min(nslot, nst);
        const int fstep = nfill > kFillAlone ? NCW : 1;
        if (lane == 0 && (fstep > 1 || warp == 0) && !*abort_flag) {
            for (int k = warp; k < nfill; k += fstep) {
                const int slot = (kbase + k) % nslot;
                const int gk = base0 + k * GS;
                const int pi = (gk >> 3) - pg0;
                tag[slot] = kbase + k;
                issue_stage<D_H, R, D_R, HG, GS>(&tm_sK, &tm_sV, &tm_zK, &tm_zV, a, smem_s + slot * stage_bytes,
                                                 smem_u32(&full[slot]), &meta[slot], l,
                                                 pi < kPageCache ? pages[pi] : bt_row[pg0 + pi], gk, hbase, HL, pol,
                                                 pol_s);
                ++nissued[slot];
            }
        }
        if (threadIdx.x == 0) {
            // every thread has read this segment's descriptor (before the barrier above):
            // step to the next one while this one streams (after an expired wait too, so
            // that the walk ends)
            ctl->advance(a.seg_table);
        }
        if (!qt_ready) {
            pdl_wait();  // q~ written by the absorb kernel
            qt_ready = true;
        }

        // This lane's q~ row, chunk-rotated so that z rows are read conflict-free: from the
        // absorb kernel's fp32 output, or as bf16 straight from the caller (absorbed weights).
        float qt[R];
        if (a.qt_in) {
            const uint4* qrow = reinterpret_cast<const uint4*>(a.qt_in + l * a.ls_qt +
                                                                 ((size_t)bb * H + hbase + (hz_ok ? hzh : 0)) * R);
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                const uint4 x = qrow[(cc + rot) % NC];
                qt[cc * 8 + 0] = hz_ok ? bf16lo(x.x) : 0.f;
                qt[cc * 8 + 1] = hz_ok ? bf16hi(x.x) : 0.f;
                qt[cc * 8 + 2] = hz_ok ? bf16lo(x.y) : 0.f;
                qt[cc * 8 + 3] = hz_ok ? bf16hi(x.y) : 0.f;
                qt[cc * 8 + 4] = hz_ok ? bf16lo(x.z) : 0.f;
                qt[cc * 8 + 5] = hz_ok ? bf16hi(x.z) : 0.f;
                qt[cc * 8 + 6] = hz_ok ? bf16lo(x.w) : 0.f;
                qt[cc * 8 + 7] = hz_ok ? bf16hi(x.w) : 0.f;
            }
        } else {
            const float* qrow = a.qt + ((size_t)vbr * H + hbase + (hz_ok ? hzh : 0)) * R;
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                const float4* src = reinterpret_cast<const float4*>(qrow + ((cc + rot) % NC) * 8);
                const float4 x0 = src[0], x1 = src[1];
                qt[cc * 8 + 0] = hz_ok ? x0.x : 0.f;
                qt[cc * 8 + 1] = hz_ok ? x0.y : 0.f;
                qt[cc * 8 + 2] = hz_ok ? x0.z : 0.f;
                qt[cc * 8 + 3] = hz_ok ? x0.w : 0.f;
                qt[cc * 8 + 4] = hz_ok ? x1.x : 0.f;
                qt[cc * 8 + 5] = hz_ok ? x1.y : 0.f;
                qt[cc * 8 + 6] = hz_ok ? x1.z : 0.f;
                qt[cc * 8 + 7] = hz_ok ? x1.w : 0.f;
            }
        }

        // Query A fragments (heads on M): rows hA, hB; k = key feature ([q | q^R]).
        uint32_t qa[D_K / 16][4];
        {
            const uint16_t* qbase = a.q + l * a.ls_q;
            const uint32_t* qA = reinterpret_cast<const uint32_t*>(qbase + ((size_t)bb * H + hbase + hA) * D_K);
            const uint32_t* qB = reinterpret_cast<const uint32_t*>(qbase + ((size_t)bb * H + hbase + hB) * D_K);
#pragma unroll
            for (int kk = 0; kk < D_K / 16; ++kk) {
                qa[kk][0] = hA < HL ? qA[kk * 8 + tq] : 0u;
                qa[kk][1] = hB < HL ? qB[kk * 8 + tq] : 0u;
                qa[kk][2] = hA < HL ? qA[kk * 8 + 4 + tq] : 0u;
                qa[kk][3] = hB < HL ? qB[kk * 8 + 4 + tq] : 0u;
            }
        }

        float o[D_H / 8][4];
#pragma unroll
        for (int n = 0; n < D_H / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float accz[R];
#pragma unroll
        for (int i = 0; i < R; ++i) accz[i] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        // After an expired wait every consumer keeps walking its loops (so all of
        // them still meet at the named barriers) but skips the work.
        for (int j = grp; j < nst; j += a.ng) {
            const int kk = kbase + j;
            const int slot = kk % nslot;
            // Abort and wait outcomes are made warp-uniform: the stage's work below is
            // warp-collective (ldmatrix, mma.sync, shuffles).
            if (__any_sync(0xffffffffu, *abort_flag != 0)) continue;
            // Groups run at different speeds, so the slot may still hold a stage one or
            // more ring rounds older than kk; its barrier parity alone cannot tell them
            // apart.  Wait until stage kk has been issued into the slot, then for its data.
            const bool ready = wait_tag(tag + slot, kk, a.status, a.wait_ns) &&
                               mbar_wait_for(smem_u32(&full[slot]), (kk / nslot) & 1, a.status, a.wait_ns);
            if (!__all_sync(0xffffffffu, ready)) {
                *abort_flag = 1;
                continue;
            }
            const uint32_t st = smem_s + slot * stage_bytes;
            const int gfirst = base0 + j * GS;  // the stage's first granule (GS-aligned)
#pragma unroll 1
            for (int sub = 0; sub < GS; ++sub) {
                const int gi = gfirst + sub;
                if (GS > 1 && (gi < sg0 || gi >= sg1)) continue;  // a granule of a neighbouring segment
                const int t0 = gi * kGran;
                const int nvalid = meta[slot] ? min(kGran, L - t0) : 0;
                // granule `sub` of the stage: rows 8 sub .. 8 sub + 7 of every 64-column part (parts
                // GS KB apart), tokens 8 sub .. 8 sub + 7 of the latents
                const uint32_t sK_s = st + sub * 1024, sV_s = st + 16 * D_K * GS + sub * 1024;
                const uint8_t* zK_p = smem + slot * stage_bytes + 16 * GS * (D_K + D_H) + sub * 16 * HL * R;
                const uint8_t* zV_p = zK_p + 16 * GS * HL * R;

                // --- shared logits [q | q^R] . [s^K | k^R] (tensor cores): 16 heads x 8 tokens
                // (two accumulators, even and odd 16-wide k chunks, halve the dependent MMA chain)
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                float c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk2 = 0; kk2 < D_K / 16; kk2 += 2) {
                    const int chunk16 = kk2 * 2 + (lane >> 3);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(sw128(sK_s + (chunk16 >> 3) * (GS * 1024), lane & 7, chunk16 & 7), b0, b1, b2, b3);
                    mma_16816(c, qa[kk2], b0, b1);
                    mma_16816(c2, qa[kk2 + 1], b2, b3);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) c[i] += c2[i];

                // --- residual logits q~ . z^K (CUDA cores): lane = (head hz, tokens half*4 .. +3)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = half * 4 + i;
                    float acc = 0.f;
                    if (hz_ok && t < nvalid) {
                        const uint4* row = reinterpret_cast<const uint4*>(zK_p + ((size_t)t * HL + hzh) * R * 2);
#pragma unroll
                        for (int cc = 0; cc < NC; ++cc) {
                            const uint4 v = row[(cc + rot) % NC];
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
                    SZ[sidx(hz, t)] = acc;
                }
                __syncwarp();

                // --- scores, mask, online softmax (rows hA: c0,c1; hB: c2,c3; tokens 2tq, 2tq+1)
                const int ta = 2 * tq, tb = 2 * tq + 1;
                float s0 = (ta < nvalid) ? (c[0] + SZ[sidx(g, ta)]) * a.scale_log2 : -INFINITY;
                float s1 = (tb < nvalid) ? (c[1] + SZ[sidx(g, tb)]) * a.scale_log2 : -INFINITY;
                float s2 = (ta < nvalid) ? (c[2] + SZ[sidx(g + 8, ta)]) * a.scale_log2 : -INFINITY;
                float s3 = (tb < nvalid) ? (c[3] + SZ[sidx(g + 8, tb)]) * a.scale_log2 : -INFINITY;
                float mx0 = fmaxf(s0, s1), mx1 = fmaxf(s2, s3);
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
                const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
                const float p0 = (mn0 == -INFINITY) ? 0.f : exp2f(s0 - mn0);
                const float p1 = (mn0 == -INFINITY) ? 0.f : exp2f(s1 - mn0);
                const float p2 = (mn1 == -INFINITY) ? 0.f : exp2f(s2 - mn1);
                const float p3 = (mn1 == -INFINITY) ? 0.f : exp2f(s3 - mn1);
                m0 = mn0;
                m1 = mn1;
                l0 = l0 * al0 + p0 + p1;
                l1 = l1 * al1 + p2 + p3;
#pragma unroll
                for (int n = 0; n < D_H / 8; ++n) {
                    o[n][0] *= al0;
                    o[n][1] *= al0;
                    o[n][2] *= al1;
                    o[n][3] *= al1;
                }
                SP[sidx(g, ta)] = p0;
                SP[sidx(g, tb)] = p1;
                SP[sidx(g + 8, ta)] = p2;
                SP[sidx(g + 8, tb)] = p3;
                if (tq == 0) {
                    SA[g] = al0;
                    SA[g + 8] = al1;
                }
                __syncwarp();

                // --- residual values p . z^V (CUDA cores)
                {
                    const float al = SA[hz];
#pragma unroll
                    for (int i = 0; i < R; ++i) accz[i] *= al;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = half * 4 + i;
                        if (hz_ok && t < nvalid) {
                            const float p = SP[sidx(hz, t)];
                            const uint4* row = reinterpret_cast<const uint4*>(zV_p + ((size_t)t * HL + hzh) * R * 2);
#pragma unroll
                            for (int cc = 0; cc < NC; ++cc) {
                                const uint4 v = row[(cc + rot) % NC];
                                accz[cc * 8 + 0] = fmaf(p, bf16lo(v.x), accz[cc * 8 + 0]);
                                accz[cc * 8 + 1] = fmaf(p, bf16hi(v.x), accz[cc * 8 + 1]);
                                accz[cc * 8 + 2] = fmaf(p, bf16lo(v.y), accz[cc * 8 + 2]);
                                accz[cc * 8 + 3] = fmaf(p, bf16hi(v.y), accz[cc * 8 + 3]);
                                accz[cc * 8 + 4] = fmaf(p, bf16lo(v.z), accz[cc * 8 + 4]);
                                accz[cc * 8 + 5] = fmaf(p, bf16hi(v.z), accz[cc * 8 + 5]);
                                accz[cc * 8 + 6] = fmaf(p, bf16lo(v.w), accz[cc * 8 + 6]);
                                accz[cc * 8 + 7] = fmaf(p, bf16hi(v.w), accz[cc * 8 + 7]);
                            }
                        }
                    }
                }

                // --- shared values p . s^V (tensor cores): P (16 heads x 8 tokens) . s^V (8 tokens x D_H)
                {
                    const uint32_t pa0 = pack_bf16x2(p0, p1), pa1 = pack_bf16x2(p2, p3);
                    const uint32_t mlo = (ta < nvalid) ? 0x0000ffffu : 0u;
                    const uint32_t mhi = (tb < nvalid) ? 0xffff0000u : 0u;
                    const uint32_t msk = mlo | mhi;  // zero s^V of masked tokens (0 * NaN guard)
#pragma unroll
                    for (int q4 = 0; q4 < D_H / 32; ++q4) {
                        const int chunk16 = q4 * 4 + (lane >> 3);
                        uint32_t v0, v1, v2, v3;
                        ldmatrix_x4_trans(sw128(sV_s + (chunk16 >> 3) * (GS * 1024), lane & 7, chunk16 & 7), v0, v1, v2, v3);
                        mma_1688(o[q4 * 4 + 0], pa0, pa1, v0 & msk);
                        mma_1688(o[q4 * 4 + 1], pa0, pa1, v1 & msk);
                        mma_1688(o[q4 * 4 + 2], pa0, pa1, v2 & msk);
                        mma_1688(o[q4 * 4 + 3], pa0, pa1, v3 & msk);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                // Release; the last of the HT warps reading this stage refills the slot
                // with the stage nslot positions ahead in this segment.
                __threadfence_block();
                if (atomicAdd(&rel[slot], 1) == HT - 1) {
                    rel[slot] = 0;
                    __threadfence_block();
                    const int jn = j + nslot;
                    if (jn < nst && !*abort_flag) {
                        const int gn = base0 + jn * GS;
                        const int pi = (gn >> 3) - pg0;
                        tag[slot] = kk + nslot;
                        issue_stage<D_H, R, D_R, HG, GS>(&tm_sK, &tm_sV, &tm_zK, &tm_zV, a, st, smem_u32(&full[slot]),
                                                         &meta[slot], l, pi < kPageCache ? pages[pi] : bt_row[pg0 + pi],
                                                         gn, hbase, HL, pol, pol_s);
                        ++nissued[slot];
                    }
                }
            }
        }
        kbase += nst;

        // --- this group's state: m, l (log2 domain), o (rows hA, hB), accz (row hzh)
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
        for (int i = 0; i < R; ++i) accz[i] += __shfl_xor_sync(0xffffffffu, accz[i], 16);

        // Groups write their state into the idle ring (or straight to the workspace
        // when there is one group), then all consumers merge it per head.
        named_bar(1, nct);  // every stage of this segment consumed: the ring is idle
        const bool direct = (a.ng == 1);
        // Workspace partials are laid out [head][slot][...] so that the combine reads
        // one head's partials contiguously.  The shared-memory staging is [group][head][WS]
        // behind the [group][head] (m, l) pairs (offset rounded to 16 bytes): rows WS floats
        // apart, 8 or 24 banks, so the fragment stores below are free of bank conflicts.
        const size_t hs_ml = direct ? (size_t)a.pmax * 2 : 2;     // stride between heads
        const size_t hs_acc = direct ? (size_t)a.pmax * W : WS;
        float* const sml_base = reinterpret_cast<float*>(smem);
        float* const sacc_base = sml_base + ((a.ng * HL * 2 + 3) & ~3);
        // (workspace rows are indexed by the global head, the staging by the group's own)
        float* gml = direct ? a.part_ml + (size_t)pslot * 2 + (size_t)hbase * hs_ml : sml_base + (size_t)grp * HL * 2;
        float* gacc = direct ? a.part_acc + (size_t)pslot * W + (size_t)hbase * hs_acc
                             : sacc_base + (size_t)grp * HL * WS;
        if (tq == 0) {
            if (hA < HL) *reinterpret_cast<float2*>(gml + hA * hs_ml) = make_float2(m0, l0);
            if (hB < HL) *reinterpret_cast<float2*>(gml + hB * hs_ml) = make_float2(m1, l1);
        }
#pragma unroll
        for (int n = 0; n < D_H / 8; ++n) {
            const int dcol = n * 8 + 2 * tq;
            if (hA < HL) *reinterpret_cast<float2*>(gacc + (size_t)hA * hs_acc + dcol) = make_float2(o[n][0], o[n][1]);
            if (hB < HL) *reinterpret_cast<float2*>(gacc + (size_t)hB * hs_acc + dcol) = make_float2(o[n][2], o[n][3]);
        }
        if (half == 0 && hz_ok) {
            float* dst = gacc + (size_t)hzh * hs_acc + D_H;
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                float4* d4 = reinterpret_cast<float4*>(dst + ((cc + rot) % NC) * 8);
                d4[0] = make_float4(accz[cc * 8 + 0], accz[cc * 8 + 1], accz[cc * 8 + 2], accz[cc * 8 + 3]);
                d4[1] = make_float4(accz[cc * 8 + 4], accz[cc * 8 + 5], accz[cc * 8 + 6], accz[cc * 8 + 7]);
            }
        }
        if (!direct) {
            // Merge the groups' states per head: first each head's merged (M, L) and every
            // group's weight 2^(m_g - M) (0 for a group that saw no token), then the
            // accumulators, four columns per thread, with all groups' loads issued together.
            named_bar(1, nct);
            const int ng = a.ng;
            const float* sml = sml_base;
            const float* sacc = sacc_base;
            float* swt = sacc_base + (size_t)ng * HL * WS;  // [group][head] weights
            float* pml = a.part_ml + (size_t)pslot * 2 + (size_t)hbase * a.pmax * 2;
            float* pacc = a.part_acc + (size_t)pslot * W + (size_t)hbase * a.pmax * W;
            for (int h = threadIdx.x; h < HL; h += nct) {
                float mg[kMaxGroups];
                float M = -INFINITY;
#pragma unroll
                for (int gg = 0; gg < kMaxGroups; ++gg) {
                    mg[gg] = gg < ng ? sml[(gg * HL + h) * 2] : -INFINITY;
                    M = fmaxf(M, mg[gg]);
                }
                float Ls = 0.f;
#pragma unroll
                for (int gg = 0; gg < kMaxGroups; ++gg) {
                    if (gg < ng) {
                        const float wg = (mg[gg] == -INFINITY) ? 0.f : exp2f(mg[gg] - M);
                        swt[gg * HL + h] = wg;
                        Ls = fmaf(wg, sml[(gg * HL + h) * 2 + 1], Ls);
                    }
                }
                *reinterpret_cast<float2*>(pml + (size_t)h * a.pmax * 2) = make_float2(M, Ls);
            }
            named_bar(1, nct);
            constexpr int W4 = W / 4;
            for (int i4 = threadIdx.x; i4 < HL * W4; i4 += nct) {
                const int h = i4 / W4, c4 = i4 - h * W4;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int gg = 0; gg < kMaxGroups; ++gg) {
                    if (gg < ng) {
                        const float4 x = *reinterpret_cast<const float4*>(sacc + ((size_t)gg * HL + h) * WS + c4 * 4);
                        const float wg = swt[gg * HL + h];
                        v.x = fmaf(wg, x.x, v.x);
                        v.y = fmaf(wg, x.y, v.y);
                        v.z = fmaf(wg, x.z, v.z);
                        v.w = fmaf(wg, x.w, v.w);
                    }
                }
                *reinterpret_cast<float4*>(pacc + (size_t)h * a.pmax * W + c4 * 4) = v;
            }
        }
    }
    // The combine kernel may now be scheduled; it waits for this grid to finish.
    pdl_trigger();
    // After an expired wait, make sure no copy is still landing in shared memory
    // before the CTA exits: wait (bounded, always with the full limit) for the last
    // phase issued into each slot.
    named_bar(1, nct);
    if (threadIdx.x == 0 && *abort_flag)
        for (int sl = 0; sl < nslot; ++sl)
            if (nissued[sl] > 0) mbar_wait(smem_u32(&full[sl]), (nissued[sl] - 1) & 1, a.status);
}

// ------------------------------------------------------------------ kernel 2
// Log-sum-exp merge of a sequence's partials, residual up-projection, bf16 store.
// grid (H, layers * B); block = NSL partial slices x W/4 column quads, one float4 of the
// accumulator row per thread.  NSL (at least ceil(D_H / (W/4)), so that every output column
// has a thread) is chosen on the host so that the grid is about one wave and most slices hold
// at most PPS partials: each slice merges its partials with all loads of a round issued
// together, then the slices are merged in shared memory; B_h^V rows are prefetched up front.
template <int D_H, int R>
__global__ void __launch_bounds__(512, 2) decode_combine_kernel(const DecodeArgs a) {
    // The next call's absorb kernel may be scheduled now: it waits for this grid to end before
    // it reads anything (an ordinary launch after this one keeps the full stream order).
    pdl_trigger();
    constexpr int W = D_H + R;
    constexpr int W4 = W / 4;
    constexpr int NSL_MAX = 512 / W4;  // slices at most
    constexpr int PPS = 6;             // partials a slice loads per round
    const int NSL = blockDim.x / W4;   // slices of this launch
    const int h = blockIdx.x, vb = blockIdx.y, tid = threadIdx.x;
    const int ly = vb / a.B, bb = vb - (vb / a.B) * a.B;
    const int H = a.H;
    __shared__ float sm_m[NSL_MAX], sm_l[NSL_MAX];
    __shared__ __align__(16) float sm_acc[NSL_MAX][W];
    __shared__ __align__(16) uint16_t sm_bv[D_H * R];  // B_h^V
    const int sl = tid / W4, c4 = tid - (tid / W4) * W4;

    // B_h^V, copied into shared memory asynchronously while the partials are loaded
    if (!a.fused_out && !a.part_out) {  // (no B^V in the fused form, nor for partials out)
        const uint16_t* bv = a.BV + ly * a.ls_BV + (size_t)h * D_H * R;
        for (int i = tid; i < D_H * R / 8; i += blockDim.x)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sm_bv + i * 8)), "l"(bv + i * 8)
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    const int L = a.seq_lens[bb];
    pdl_wait();
    const int OW = a.fused_out ? W : D_H;  // output row width
    uint16_t* dst = a.out + ly * a.ls_out + ((size_t)bb * H + h) * OW;
    float* pdst = a.part_out ? a.part_out + ((size_t)bb * H + h) * (W + 2) : nullptr;
    if (L < 1 || L > a.max_pages * kBlockSize) {
        // partials out: a sequence with no tokens in this range is an empty partial, not an error
        if (tid == 0 && h == 0 && !(pdst && L == 0)) set_status(a.status, LRKV_DEV_BAD_SEQLEN);
        if (pdst) {
            for (int i = tid; i < W + 2; i += blockDim.x) pdst[i] = i == W ? -INFINITY : 0.f;
        } else {
            for (int i = tid; i < OW; i += blockDim.x) dst[i] = 0;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        return;
    }
    // partial slots first .. first + np - 1, recorded by the split kernel
    const int2 fe = a.seg_table[vb * a.nhg + h / (H / a.nhg)];
    const int first = fe.x, np = fe.y;
    const float* pml = a.part_ml + ((size_t)h * a.pmax + first) * 2;
    const float4* pacc = reinterpret_cast<const float4*>(a.part_acc + ((size_t)h * a.pmax + first) * W);

    {
        float m = -INFINITY, l = 0.f;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p0 = sl; p0 < np; p0 += NSL * PPS) {
            float2 ml[PPS];
            float4 x[PPS];
#pragma unroll
            for (int u = 0; u < PPS; ++u) {
                const int p = p0 + u * NSL;
                ml[u] = p < np ? *reinterpret_cast<const float2*>(pml + 2 * p) : make_float2(-INFINITY, 0.f);
                x[u] = p < np ? pacc[(size_t)p * W4 + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mn = m;
#pragma unroll
            for (int u = 0; u < PPS; ++u) mn = fmaxf(mn, ml[u].x);
            if (mn != -INFINITY) {
                const float sc = (m == -INFINITY) ? 0.f : exp2f(m - mn);
                l *= sc;
                v.x *= sc;
                v.y *= sc;
                v.z *= sc;
                v.w *= sc;
#pragma unroll
                for (int u = 0; u < PPS; ++u) {
                    const float w = (ml[u].x == -INFINITY) ? 0.f : exp2f(ml[u].x - mn);
                    l = fmaf(w, ml[u].y, l);
                    v.x = fmaf(w, x[u].x, v.x);
                    v.y = fmaf(w, x[u].y, v.y);
                    v.z = fmaf(w, x[u].z, v.z);
                    v.w = fmaf(w, x[u].w, v.w);
                }
                m = mn;
            }
        }
        *reinterpret_cast<float4*>(&sm_acc[sl][c4 * 4]) = v;
        if (c4 == 0) {
            sm_m[sl] = m;
            sm_l[sl] = l;
        }
    }
    __syncthreads();
    if (tid < W4) {
        float M = -INFINITY;
        for (int i = 0; i < NSL; ++i) M = fmaxf(M, sm_m[i]);  // (NSL is known at run time only)
        float lsum = 0.f;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < NSL; ++i) {
            const float w = (sm_m[i] == -INFINITY) ? 0.f : exp2f(sm_m[i] - M);
            const float4 x = *reinterpret_cast<const float4*>(&sm_acc[i][tid * 4]);
            lsum = fmaf(w, sm_l[i], lsum);
            v.x = fmaf(w, x.x, v.x);
            v.y = fmaf(w, x.y, v.y);
            v.z = fmaf(w, x.z, v.z);
            v.w = fmaf(w, x.w, v.w);
        }
        if (pdst) {  // unnormalised: the merge over token ranges normalises
            pdst[tid * 4] = v.x;
            pdst[tid * 4 + 1] = v.y;
            pdst[tid * 4 + 2] = v.z;
            pdst[tid * 4 + 3] = v.w;
            if (tid == 0) {
                pdst[W] = M;
                pdst[W + 1] = lsum;
            }
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const float4 r = lsum > 0.f ? make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        // each thread reads only its own quad, so slice 0's slot can take the result
        *reinterpret_cast<float4*>(&sm_acc[0][tid * 4]) = r;
        if (a.fused_out) {  // [o_s | o_z] / l: the B^V up-projection belongs to the caller's W^O
            const float rr[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const __nv_bfloat16 ob = __float2bfloat16_rn(rr[k]);
                dst[tid * 4 + k] = *reinterpret_cast<const uint16_t*>(&ob);
            }
        }
    }
    if (a.fused_out || pdst) return;
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (tid < D_H) {
        float v = sm_acc[0][tid];
        const uint4* bvr = reinterpret_cast<const uint4*>(sm_bv + tid * R);
#pragma unroll
        for (int i = 0; i < R / 8; ++i) {
            const uint4 q = bvr[i];
            v = fmaf(bf16lo(q.x), sm_acc[0][D_H + i * 8 + 0], v);
            v = fmaf(bf16hi(q.x), sm_acc[0][D_H + i * 8 + 1], v);
            v = fmaf(bf16lo(q.y), sm_acc[0][D_H + i * 8 + 2], v);
            v = fmaf(bf16hi(q.y), sm_acc[0][D_H + i * 8 + 3], v);
            v = fmaf(bf16lo(q.z), sm_acc[0][D_H + i * 8 + 4], v);
            v = fmaf(bf16hi(q.z), sm_acc[0][D_H + i * 8 + 5], v);
            v = fmaf(bf16lo(q.w), sm_acc[0][D_H + i * 8 + 6], v);
            v = fmaf(bf16hi(q.w), sm_acc[0][D_H + i * 8 + 7], v);
        }
        const __nv_bfloat16 ob = __float2bfloat16_rn(v);
        dst[tid] = *reinterpret_cast<const uint16_t*>(&ob);
    }
}

// Merge of decode partials over parts of the sequences' token ranges (each part, e.g. the
// cache shard of one device, decoded with partials out): log-sum-exp over the parts,
//   M = max_p m_p,  w_p = 2^(m_p - M),  acc = sum_p w_p acc_p,  l = sum_p w_p l_p,
//   out = (acc_s + B_h^V acc_z) / l,
// i.e. the combine's merge with the parts in place of the splits.  grid (H, B), one thread per
// accumulator column.
template <int D_H, int R>
__global__ void __launch_bounds__(256) decode_merge_kernel(const float* parts, int nparts, const uint16_t* BV,
                                                           int B, int H, uint16_t* out, uint32_t* status) {
    constexpr int W = D_H + R, PW = W + 2;
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    __shared__ float sacc[W];
    __shared__ float sl;
    const size_t pstride = (size_t)B * H * PW;  // between parts
    const float* p0 = parts + ((size_t)b * H + h) * PW;
    float M = -INFINITY;
    for (int p = 0; p < nparts; ++p) M = fmaxf(M, p0[p * pstride + W]);
    float l = 0.f, acc = 0.f;
    for (int p = 0; p < nparts; ++p) {
        const float* row = p0 + p * pstride;
        const float m = row[W];
        const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
        l = fmaf(w, row[W + 1], l);
        if (tid < W) acc = fmaf(w, row[tid], acc);
    }
    if (tid < W) sacc[tid] = acc;
    if (tid == 0) {
        sl = l;
        if (!(l > 0.f)) set_status(status, LRKV_DEV_BAD_SEQLEN);  // no part held a token of it
    }
    __syncthreads();
    if (tid < D_H) {
        float v = sacc[tid];
        const uint16_t* bv = BV + ((size_t)h * D_H + tid) * R;
#pragma unroll
        for (int j = 0; j < R; ++j) v = fmaf(__uint_as_float((uint32_t)bv[j] << 16), sacc[D_H + j], v);
        const float inv = sl > 0.f ? 1.f / sl : 0.f;
        const __nv_bfloat16 ob = __float2bfloat16_rn(v * inv);
        out[((size_t)b * H + h) * D_H + tid] = *reinterpret_cast<const uint16_t*>(&ob);
    }
}

cudaError_t launch_decode_merge(const float* parts, int nparts, const uint16_t* BV, int B, int H, int d_h, int r,
                                uint16_t* out, uint32_t* status, cudaStream_t stream) {
#define LRKV_MERGE(DH, RR)                                                                                    \
    if (d_h == DH && r == RR) {                                                                               \
        decode_merge_kernel<DH, RR><<<dim3(H, B), 256, 0, stream>>>(parts, nparts, BV, B, H, out, status);   \
        return cudaGetLastError();                                                                            \
    }
    LRKV_MERGE(64, 8) LRKV_MERGE(64, 16) LRKV_MERGE(64, 32) LRKV_MERGE(128, 8) LRKV_MERGE(128, 16)
    LRKV_MERGE(128, 32)
#undef LRKV_MERGE
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ host side
struct DecodePlan {
    int ng, nslot, stage_bytes, smem_bytes, threads, gpst;
};

static int decode_fixed_smem(int ncw, int nslot) {
    return nslot * 8 + ((4 * nslot + 3) & ~3) * 4 + (kPageCache + kSeqCache) * 4 + ncw * kScratchFloats * 4 + 16 +
           kCtlBytes + 1024;  // (the abort flag; the control block; alignment of the ring)
}

int decode_head_groups(int H, int R) {
    if (H * R <= kGroupLatents) return 1;
    for (int g = 2; g <= 8; g *= 2)
        if (H % g == 0 && (H / g) * R <= kGroupLatents && ((H / g) * R) % 128 == 0) return g;
    return 1;
}

int decode_stage_granules(int H, int D_H, int R, int D_R) {
    if (decode_head_groups(H, R) > 1) return 1;
    const int gran_bytes = 16 * (2 * D_H + D_R) + 32 * H * R;
    return 2 * gran_bytes <= kSmallStageBytes ? 2 : 1;
}

DecodePlan decode_plan(int H_all, int D_H, int R, int D_R, int smem_limit) {
    DecodePlan p{};
    const int H = H_all / decode_head_groups(H_all, R);  // heads of one CTA's group
    const int HT = (H + 15) / 16;
    p.gpst = decode_stage_granules(H_all, D_H, R, D_R);
    p.stage_bytes = ((p.gpst * (16 * (2 * D_H + D_R) + 32 * H * R)) + 1023) & ~1023;
    int nslot = 16;
    while (nslot > 2 && nslot * p.stage_bytes + decode_fixed_smem(8, nslot) > smem_limit) --nslot;
    p.nslot = nslot;
    int ng = max(1, min(8 / HT, nslot - 2));
    // the group merge reuses the ring: ng * H * (WS + 3) floats (+ 3 of alignment) must fit in it
    const int WS = decode_stage_stride(D_H + R);
    while (ng > 1 && ((size_t)ng * H * (WS + 3) + 3) * 4 > (size_t)nslot * p.stage_bytes) --ng;
    p.ng = ng;
    p.threads = 32 * HT * ng;
    p.smem_bytes = nslot * p.stage_bytes + decode_fixed_smem(HT * ng, nslot);
    return p;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool decode_fits(int H, int D_H, int R, int D_R, int smem_limit) {
    const DecodePlan p = decode_plan(H, D_H, R, D_R, smem_limit);
    return p.smem_bytes <= smem_limit;
}

size_t decode_workspace_bytes(int H, int D_H, int R, int nvb, int nranges) {
    const size_t nseg = (size_t)nvb * decode_head_groups(H, R);  // virtual sequences of the scan
    const size_t pmax = nseg + (size_t)nranges;
    return align256(pmax * H * 2 * sizeof(float)) + align256(pmax * H * (D_H + R) * sizeof(float)) +
           align256((size_t)nvb * H * R * sizeof(float)) + align256(nseg * sizeof(int2));
}

void decode_carve_workspace(DecodeArgs* a, void* ws, int H, int D_H, int R, int nvb, int nranges) {
    const size_t pmax = (size_t)nvb * decode_head_groups(H, R) + (size_t)nranges;
    uint8_t* base = static_cast<uint8_t*>(ws);
    a->part_ml = reinterpret_cast<float*>(base);
    base += align256(pmax * H * 2 * sizeof(float));
    a->part_acc = reinterpret_cast<float*>(base);
    base += align256(pmax * H * (D_H + R) * sizeof(float));
    a->qt = reinterpret_cast<float*>(base);
    base += align256((size_t)nvb * H * R * sizeof(float));
    a->seg_table = reinterpret_cast<int2*>(base);
    a->pmax = (int)pmax;
}

template <typename... Args>
static cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D_H, int R>
static cudaError_t launch_combine(const DecodeArgs& a, int nvb, int sms, cudaStream_t stream) {
    // Slices per (head, sequence): enough threads for about one wave of the GPU in total, and at
    // least one thread per output column.
    constexpr int W4 = (D_H + R) / 4;
    const long long pairs = (long long)a.H * nvb;
    const int nsl_min = (D_H + W4 - 1) / W4;
    const int nsl = (int)max((long long)nsl_min,
                             min((long long)(512 / W4), ((long long)sms * 1024) / max(1LL, pairs * W4)));
    return launch_pdl(decode_combine_kernel<D_H, R>, dim3(a.H, nvb), dim3(nsl * W4), 0, stream, a);
}

template <int D_H, int R, int D_R>
static cudaError_t launch_decode_t(const CUtensorMap& tK, const CUtensorMap& tV, const CUtensorMap& tZK,
                                   const CUtensorMap& tZV, DecodeArgs a, const DecodePlan& p, int sms,
                                   cudaStream_t stream) {
    // Head groups occur only where a token's latents for all heads exceed kGroupLatents elements,
    // which with H <= 128 needs r = 32.
    auto split = a.gpst == 2 ? decode_split_kernel<D_H, R, D_R, false, 2> : decode_split_kernel<D_H, R, D_R, false, 1>;
    if constexpr (R * 128 > kGroupLatents) {
        if (a.nhg > 1) split = decode_split_kernel<D_H, R, D_R, true, 1>;
    }
    cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    const int nvb = a.layers * a.B;
    const int grid = a.nranges < sms ? a.nranges : sms;
    // 128 heads of d_h = 128: the scan on the 5th-generation tensor cores (heads = the MMAs' M)
    if constexpr (D_H == 128 && D_R == 0 && (R == 8 || R == 16)) {
        if (a.H == 128 && a.nhg == 1 && a.gpst == 1) {
            if (!a.qt_in) {
                e = launch_pdl(decode_absorb_kernel<D_H, R, D_R>, dim3(a.H, nvb), dim3(256), 0, stream, a);
                if (e != cudaSuccess) return e;
            }
            e = launch_decode_tc_split<R>(tK, tV, a, grid, decode_tc_smem_bytes(p.nslot, p.stage_bytes), !a.qt_in,
                                          stream);
            if (e != cudaSuccess) return e;
            return launch_combine<D_H, R>(a, nvb, sms, stream);
        }
    }
    if (a.qt_in) {
        // q~ comes from the caller: no absorb kernel, and the split is an ordinary launch --
        // a dependent launch could start streaming the cache before the caller's previous
        // kernel on this stream (an append of the newest rows) has finished.
        split<<<grid, p.threads, p.smem_bytes, stream>>>(tK, tV, tZK, tZV, a);
        e = cudaGetLastError();
    } else {
        e = launch_pdl(decode_absorb_kernel<D_H, R, D_R>, dim3(a.H, nvb), dim3(256), 0, stream, a);
        if (e != cudaSuccess) return e;
        e = launch_pdl(split, dim3(grid), dim3(p.threads), p.smem_bytes, stream, tK, tV, tZK, tZV, a);
    }
    if (e != cudaSuccess) return e;
    return launch_combine<D_H, R>(a, nvb, sms, stream);
}

cudaError_t launch_decode(const CUtensorMap& tK, const CUtensorMap& tV, const CUtensorMap& tZK,
                          const CUtensorMap& tZV, DecodeArgs a, int D_H, int R, int D_R, int sms, int smem_limit,
                          cudaStream_t stream) {
    const DecodePlan p = decode_plan(a.H, D_H, R, D_R, smem_limit);
    a.ng = p.ng;
    a.nslot = p.nslot;
    a.stage_bytes = p.stage_bytes;
    a.gpst = p.gpst;
    // a pipeline drain and refill at a sequence boundary costs about as long as streaming
    // 128 KB through one SM (~3 us)
    a.bubble = ((128 << 10) * p.gpst + p.stage_bytes - 1) / p.stage_bytes;  // (in granules)
#define LRKV_DEC(DH, RR)                                                                     \
    if (D_H == DH && R == RR)                                                                \
        return D_R == 0 ? launch_decode_t<DH, RR, 0>(tK, tV, tZK, tZV, a, p, sms, stream)    \
                        : launch_decode_t<DH, RR, 64>(tK, tV, tZK, tZV, a, p, sms, stream);
    LRKV_DEC(64, 8) LRKV_DEC(64, 16) LRKV_DEC(64, 32) LRKV_DEC(128, 8) LRKV_DEC(128, 16) LRKV_DEC(128, 32)
#undef LRKV_DEC
    return cudaErrorInvalidValue;
}

}  // namespace lrkv
