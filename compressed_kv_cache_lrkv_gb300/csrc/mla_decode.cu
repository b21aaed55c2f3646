// mla_decode.cu -- multi-head latent attention decode with absorbed weights on the
// 5th-generation tensor cores ("Embeddings II: MLA & Architectural Choices": weight
// absorption, decoupled RoPE, the softmax denominator of the concatenated width; the
// associative form of "Low-Rank Key Value Attention", backup frame "MLA also admits
// associative computation").
//
// Per token the cache holds one row [c_t | k^R_t] (latent d_c = 512, positional key
// d_rope = 64), shared by all heads.  With W^UK folded into the query and W^UV into the
// output projection, head i computes
//     logit_{i,t} = [q~_i | q^R_i] . [c_t | k^R_t] * scale,   o_i = sum_t p_{i,t} c_t.
// That is multi-query attention with 128 query rows per token: ~242 flop per cached byte,
// so both contractions run on tcgen05 (heads on M = 128, 64-token tiles = one page).
//
// A 512-column fp32 accumulator for 128 heads fills all of TMEM, and Q (128 x 576 bf16)
// alone takes 144 KiB of shared memory, so one split is handled by a cluster of two CTAs
// that divide the columns: rank r owns c[256r, 256r + 256) and k^R[32r, 32r + 32).  Each
// CTA loads only its columns of Q and of every page (every cached byte is read once),
// computes the partial logits S_r = Q_r K_r^T, and the two exchange S_r through
// distributed shared memory; both then hold S = S_0 + S_1 (fp32 addition commutes, so the
// two softmaxes agree bit for bit) and each accumulates its own half O_r += P V_r, with
// V_r = its 256 latent columns of the same page.  Splits write (m, l, O) partials; a
// combine kernel merges them per (sequence, head) by log-sum-exp.
//
// Warp roles per CTA: warp 0 TMA producer (Q per split, 3-stage page ring), warp 1 score
// MMAs and TMEM owner, warp 2 P.V MMAs, warps 3-6 softmax (one head row per thread, TMEM
// lane quarter = warp % 4), warps 7-10 senders (the same rows' partial logits to the peer,
// one tile ahead of the softmax, so the transfer overlaps it).  Every wait is bounded; an expired wait sets
// LRKV_DEV_TIMEOUT and the abort flag of both CTAs of the pair.
#include <type_traits>

#include "kernels.h"
#include "lrkv_internal.cuh"
#include "mla.h"

namespace lrkv {

namespace {

constexpr int kDC = 512, kDR = 64, kDK = kDC + kDR;
constexpr int kTok = 64;                        // tokens per tile (one page)
// Per CTA: four 64-column latent blocks (128-byte swizzle) and one 32-column block of k^R
// (64-byte swizzle), for Q and for every page.
constexpr uint32_t QATOM = 128 * 128;           // [128 heads][64 columns] bf16
constexpr uint32_t QHALF = 128 * 64;            // [128 heads][32 columns] bf16
constexpr uint32_t KATOM = kTok * 128;          // [64 tokens][64 columns] bf16
constexpr uint32_t KHALF = kTok * 64;           // [64 tokens][32 columns] bf16
constexpr int kStages = 3;
constexpr uint32_t STAGE = 4 * KATOM + KHALF;   // 36 KiB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_QR = 4 * QATOM;
constexpr uint32_t OFF_KV = OFF_QR + QHALF;                   // 72 KiB
constexpr uint32_t OFF_RECV = OFF_KV + kStages * STAGE;      // partial logits from the peer, [16 chunks][128 rows][16 B]
constexpr uint32_t OFF_BAR = OFF_RECV + 128 * 256;
constexpr uint32_t OFF_SEQ = OFF_BAR + 256;                  // first 256 sequence lengths
constexpr uint32_t kSmemBytes = OFF_SEQ + 1024 + 1024;
// TMEM: three 64-column partial-S buffers (one per ring stage: tile g uses buffer g % 3), then
// the 256-column O_r accumulator.
constexpr uint32_t TM_S = 0, TM_O = 3 * kTok, TM_COLS = 512;
constexpr int kThreads = 352;
constexpr float kRescaleThreshold = 8.0f;      // log2 units

static_assert(kDK == 576, "row width");
static_assert(OFF_KV % 1024 == 0 && STAGE % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
static_assert(kSmemBytes <= 232448, "shared memory");

// ---- cluster primitives
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address in the shared memory of CTA `rank` of this cluster of the variable at `local`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// Asynchronous 16-byte store into another CTA's shared memory that counts its bytes on that
// CTA's mbarrier (complete_tx), like a TMA copy: no per-store fence or arrival is needed.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w,
                                            uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
                 "r"(x), "r"(y), "r"(z), "r"(w), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster.  Relaxed: it only tells the peer that
// this CTA has consumed what the peer wrote -- the values were loaded and used before it.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait (acquire at cluster scope) for a phase completed by the peer CTA's arrivals.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint32_t* status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            set_status(status, LRKV_DEV_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Prefetch a tensor box into L2 (no shared memory, no completion tracking).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, uint32_t* status) {
    const bool ok = mbar_wait(bar, parity, status);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool wait_all_cluster(uint32_t bar, uint32_t parity, uint32_t* status) {
    const bool ok = mbar_wait_cluster(bar, parity, status);
    return __all_sync(0xffffffffu, ok);
}

// K-major 128-byte-swizzled operand descriptors: Q atoms [128][64] are 16 KiB apart, page atoms
// [64][64] 8 KiB apart; the value operand is the same page read MN-major (N = latent columns
// in 64-wide blocks 8 KiB apart, K = tokens in 8-row groups 1 KiB apart).
__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return sdesc(a, 16, 1024, 2); }
__device__ __forceinline__ uint64_t kdesc64(uint32_t a) { return sdesc(a, 16, 512, 4); }
__device__ __forceinline__ uint64_t vdesc(uint32_t a) { return sdesc(a, KATOM, 1024, 2); }

// ---- partition: a sequence's pages are cut into contiguous splits of about equal size,
// at most max(npairs, B) splits in all (every split lies inside one sequence).
struct MlaSplit {
    int b, p0, p1;
};

// Sequence lengths, the first kSeqCache from a shared-memory copy (the partition walks them
// several times per CTA).
constexpr int kSeqCache = 256;
struct Lens {
    const int32_t* g;
    const int* s;
    int B, cap;
    __device__ __forceinline__ int pages(int b) const {
        const int L = b < kSeqCache ? s[b] : g[b];
        return (L >= 1 && L <= cap) ? (L + kTok - 1) / kTok : 0;
    }
};

__device__ __forceinline__ int partition_chunk(const Lens& ln, int G, int* nsplits) {
    long long total = 0;
    for (int b = 0; b < ln.B; ++b) total += ln.pages(b);
    const int denom = G > ln.B ? G - ln.B : 1;
    const int chunk = (int)max(1LL, (total + denom - 1) / denom);
    int ns = 0;
    for (int b = 0; b < ln.B; ++b) ns += (ln.pages(b) + chunk - 1) / chunk;
    *nsplits = ns;
    return chunk;
}

__device__ __forceinline__ MlaSplit split_info(const Lens& ln, int chunk, int s) {
    int base = 0;
    for (int b = 0; b < ln.B; ++b) {
        const int gr = ln.pages(b);
        const int ns = (gr + chunk - 1) / chunk;
        if (s < base + ns) {
            const int i = s - base;
            return MlaSplit{b, (int)((long long)i * gr / ns), (int)((long long)(i + 1) * gr / ns)};
        }
        base += ns;
    }
    return MlaSplit{0, 0, 0};
}

// Score MMAs of one CTA: S_r = Q_r . K_r^T over its 16 latent K-steps and 2 positional ones.
// Tile g uses ring stage and S buffer g % 3; the tile loop branches on it so that every
// descriptor is loop-invariant.
__device__ __forceinline__ bool score_mmas(const MlaArgs& a, const Lens& ln, uint32_t S0, uint32_t tmem,
                                           uint64_t* bars, volatile int* abort_flag, int pair, int nsplits,
                                           int chunk) {
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* k_full = bars + 2;
    uint64_t* s_full = bars + 8;
    uint64_t* s_free = bars + 11;
    auto B = [&](uint64_t* p) { return smem_u32(p); };
    constexpr uint32_t id_S = idesc_bf16_f32(128, kTok);
    const uint64_t dQ = kdesc(S0 + OFF_Q), dQr = kdesc64(S0 + OFF_QR);
    const uint64_t dK = kdesc(S0 + OFF_KV), dKr = kdesc64(S0 + OFF_KV + 4 * KATOM);
    auto kq = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * QATOM + (kk & 3) * 32) >> 4); };
    auto kk_ = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * KATOM + (kk & 3) * 32) >> 4); };
    auto tile = [&](int g, auto U) -> bool {
        constexpr int st = decltype(U)::value;  // ring stage = S buffer
        // S buffer st still holds P_{g-3} until P_{g-3} . V_{g-3} has completed
        if (__any_sync(0xffffffffu, *abort_flag != 0) || !wait_all(B(k_full + st), (g / kStages) & 1, a.status) ||
            (g >= kStages && !wait_all(B(s_free + st), (g / kStages - 1) & 1, a.status)))
            return false;
        tc_fence_after();
        constexpr uint64_t so = (uint64_t)(st * STAGE) >> 4;
        const uint32_t d = tmem + TM_S + st * kTok;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            if (elect_one_sync()) tc_mma_bf16(d, dQ + kq(kk), dK + so + kk_(kk), id_S, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
            if (elect_one_sync()) tc_mma_bf16(d, dQr + (uint64_t)(kk * 2), dKr + so + (uint64_t)(kk * 2), id_S, 1);
        if (elect_one_sync()) tc_commit(B(s_full + st));
        __syncwarp();
        return true;
    };
    bool ok = true;
    int g = 0, sidx = 0;
    for (int s = pair; s < nsplits && ok; s += a.npairs, ++sidx) {
        const MlaSplit sp = split_info(ln, chunk, s);
        ok = wait_all(B(q_full), sidx & 1, a.status);
        if (ok) tc_fence_after();
        for (int p = sp.p0; p < sp.p1 && ok; ++p, ++g) {
            switch (g % kStages) {
                case 0: ok = tile(g, std::integral_constant<int, 0>{}); break;
                case 1: ok = tile(g, std::integral_constant<int, 1>{}); break;
                default: ok = tile(g, std::integral_constant<int, 2>{}); break;
            }
        }
        // Q may be replaced once every score MMA of this split has read it
        if (elect_one_sync()) tc_commit(B(q_empty));
        __syncwarp();
    }
    return ok;
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_split_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQr,
                            const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ CUtensorMap tmKVr,
                            const MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzle atoms; the offset is the same in both CTAs of the
    // pair (same kernel, same dynamic shared-memory base), so mapped addresses line up.
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t S0 = smem_u32(smem);
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int col0 = rank * 256;              // first latent column of this CTA
    const int colr = kDC + rank * (kDR / 2);  // first positional-key column of this CTA
    const int pair = blockIdx.x >> 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* q_full = bars + 0;     // Q of the split landed
    uint64_t* q_empty = bars + 1;    // score MMAs of the split done with Q
    uint64_t* k_full = bars + 2;     // [3] page landed
    uint64_t* k_empty = bars + 5;    // [3] P.V done with the page
    uint64_t* s_full = bars + 8;     // [3] partial S of tile g in TMEM buffer g % 3
    uint64_t* s_free = bars + 11;    // [3] P.V done with the P held in that S buffer
    uint64_t* p_full = bars + 14;    // softmax wrote P (128 arrivals)
    uint64_t* o_done = bars + 15;    // [3] P.V of tile g (barrier g % 3) complete
    uint64_t* recv_full = bars + 18; // the peer's partial S is in this CTA's receive buffer (1 local arrival + 32 KiB)
    uint64_t* peer_free = bars + 19; // the peer has read what this CTA wrote into its buffer (4 remote arrivals)
    uint64_t* mma_drain = bars + 20;
    uint64_t* pv_drain = bars + 21;
    uint64_t* s_read = bars + 22;    // [3] the senders have read the partial S in that buffer (128 arrivals)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 25);
    volatile int* abort_flag = reinterpret_cast<int*>(bars + 26);
    auto B = [&](uint64_t* p) { return smem_u32(p); };
    auto aborted = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0); };
    // Abort this CTA and its peer (whose loops would otherwise wait for this one).
    auto abort_pair = [&]() {
        *abort_flag = 1;
        st_cluster_u32(peer_addr(smem_u32(const_cast<int*>(abort_flag)), peer), 1u);
    };

    if (threadIdx.x == 0) {
        mbar_init(B(q_full), 1);
        mbar_init(B(q_empty), 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(B(k_full + i), 1);
            mbar_init(B(k_empty + i), 1);
            mbar_init(B(s_full + i), 1);
            mbar_init(B(s_free + i), 1);
            mbar_init(B(o_done + i), 1);
            mbar_init(B(s_read + i), 128);
        }
        mbar_init(B(p_full), 128);
        mbar_init(B(recv_full), 1);
        mbar_init(B(peer_free), 4);
        mbar_init(B(mma_drain), 1);
        mbar_init(B(pv_drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int b = threadIdx.x; b < a.B && b < kSeqCache; b += blockDim.x)
        reinterpret_cast<int*>(smem + OFF_SEQ)[b] = a.seq_lens[b];
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const Lens ln{a.seq_lens, reinterpret_cast<const int*>(smem + OFF_SEQ), a.B, a.max_pages * kTok};
    int nsplits;
    const int chunk = partition_chunk(ln, a.npairs, &nsplits);
    // one CTA publishes each sequence's first split and split count for the combine
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        int base = 0;
        for (int b = 0; b < a.B; ++b) {
            const int cnt = (ln.pages(b) + chunk - 1) / chunk;
            a.seq_first[b] = base;
            a.seq_count[b] = cnt;
            base += cnt;
        }
    }

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        const uint64_t pol = policy_evict_first();
        bool ok = true;
        int g = 0, sidx = 0, q_issued = -1;
        for (int s = pair; s < nsplits && ok; s += a.npairs, ++sidx) {
            const MlaSplit sp = split_info(ln, chunk, s);
            if ((sidx > 0 && !wait_all(B(q_empty), (sidx - 1) & 1, a.status)) || aborted()) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(B(q_full), 4 * QATOM + QHALF);
                for (int i = 0; i < 4; ++i) tma_load_3d(S0 + OFF_Q + i * QATOM, &tmQ, col0 + i * 64, 0, sp.b, B(q_full));
                tma_load_3d(S0 + OFF_QR, &tmQr, colr, 0, sp.b, B(q_full));
            }
            q_issued = sidx;
            // Physical rows of the split's pages sit in registers, 32 per batch (lane i holds
            // page p0 + 32 * batch + i), the next batch fetched one batch ahead.
            const int32_t* bt = a.block_table + (size_t)sp.b * a.max_pages;
            const int oob_row = a.num_blocks * kTok;  // whole box out of bounds -> zero fill
            auto fetch = [&](int batch) {
                const int p = sp.p0 + batch * 32 + lane;
                int row = oob_row;
                if (p < sp.p1) {
                    const int blk = bt[p];
                    if (blk >= 0 && blk < a.num_blocks)
                        row = blk * kTok;
                    else
                        set_status(a.status, LRKV_DEV_BAD_BLOCK);
                }
                return row;
            };
            int cur = fetch(0), nxt = fetch(1);
            const int npg = sp.p1 - sp.p0;
            for (int j = 0; j < npg; ++j, ++g) {
                if (j > 0 && (j & 31) == 0) {
                    cur = nxt;
                    nxt = fetch((j >> 5) + 1);
                }
                const int row = __shfl_sync(0xffffffffu, cur, j & 31);
                // the page one ring-depth ahead, into L2 now, so that its copy into the ring (issued
                // once this tile's P.V frees a stage) does not wait for HBM
                const int jp = j + kStages;
                const int prow = __shfl_sync(0xffffffffu, ((jp & ~31) == (j & ~31)) ? cur : nxt, jp & 31);
                const int st = g % kStages;
                if ((g >= kStages && !wait_all(B(k_empty + st), (g / kStages - 1) & 1, a.status)) || aborted()) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t dst = S0 + OFF_KV + st * STAGE, bar = B(k_full + st);
                    mbar_arrive_expect_tx(bar, STAGE);
                    for (int i = 0; i < 4; ++i) tma_load_2d_hint(dst + i * KATOM, &tmKV, col0 + i * 64, row, bar, pol);
                    tma_load_2d_hint(dst + 4 * KATOM, &tmKVr, colr, row, bar, pol);
                    if (jp < npg && prow < a.num_blocks * kTok) {
                        for (int i = 0; i < 4; ++i) tma_prefetch_2d(&tmKV, col0 + i * 64, prow);
                        tma_prefetch_2d(&tmKVr, colr, prow);
                    }
                }
                __syncwarp();
            }
        }
        if (!ok) {
            if (lane == 0) abort_pair();
            // let the copies still in flight land before the CTA exits
            for (int k = max(0, g - kStages); k < g; ++k) wait_all(B(k_full + k % kStages), (k / kStages) & 1, a.status);
            if (q_issued >= 0) wait_all(B(q_full), q_issued & 1, a.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- score MMAs
        const bool ok = score_mmas(a, ln, S0, tmem, bars, abort_flag, pair, nsplits, chunk);
        if (!ok && lane == 0) abort_pair();
        if (elect_one_sync()) tc_commit(B(mma_drain));
        __syncwarp();
        wait_all(B(mma_drain), 0, a.status);
    } else if (warp == 2) {
        // ---------------------------------------------------------------- P.V MMAs
        // O_r (128 heads x 256 latent columns, fp32 in TMEM) += P (TMEM, bf16) . V_r (the page's
        // latent columns of this CTA, read MN-major): four K=16 steps of N = 256.
        constexpr uint32_t id_PV = idesc_bf16_f32(128, 256) | (1u << 16);
        const uint64_t dV = vdesc(S0 + OFF_KV);
        auto pv = [&](int g, bool first, auto U) -> bool {
            constexpr int st = decltype(U)::value;  // ring stage = S buffer
            // P_g is in TMEM, and the senders are done with S_g (the buffer is freed after this P.V)
            if (aborted() || !wait_all(B(p_full), g & 1, a.status) ||
                !wait_all(B(s_read + st), (g / kStages) & 1, a.status))
                return false;
            tc_fence_after();
            constexpr uint64_t so = (uint64_t)(st * STAGE) >> 4;
            const uint32_t pt = tmem + TM_S + st * kTok;
#pragma unroll
            for (int kk = 0; kk < kTok / 16; ++kk)
                if (elect_one_sync())
                    tc_mma_bf16_ts(tmem + TM_O, pt + kk * 8, dV + so + (uint64_t)((kk * 2048) >> 4), id_PV,
                                   (first && kk == 0) ? 0u : 1u);
            if (elect_one_sync()) {
                tc_commit(B(o_done + st));
                tc_commit(B(k_empty + st));
                tc_commit(B(s_free + st));
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        int g = 0;
        for (int s = pair; s < nsplits && ok; s += a.npairs) {
            const MlaSplit sp = split_info(ln, chunk, s);
            for (int p = sp.p0; p < sp.p1 && ok; ++p, ++g) {
                const bool first = p == sp.p0;
                switch (g % kStages) {
                    case 0: ok = pv(g, first, std::integral_constant<int, 0>{}); break;
                    case 1: ok = pv(g, first, std::integral_constant<int, 1>{}); break;
                    default: ok = pv(g, first, std::integral_constant<int, 2>{}); break;
                }
            }
        }
        if (!ok && lane == 0) abort_pair();
        if (elect_one_sync()) tc_commit(B(pv_drain));
        __syncwarp();
        wait_all(B(pv_drain), 0, a.status);
    } else if (warp >= 7) {
        // ---------------------------------------------------------------- senders
        // Partial logits of tile g, rows of this warp's TMEM lane quarter, into the peer's
        // receive buffer as asynchronous stores counted on the peer's recv_full -- once the peer
        // has read tile g-1 out of it.
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const uint32_t tl = (uint32_t)(q4 * 32) << 16;
        const uint32_t peer_row = peer_addr(S0 + OFF_RECV + row * 16, peer);
        const uint32_t peer_recv_full = peer_addr(B(recv_full), peer);
        bool ok = true;
        int g = 0;
        for (int s = pair; s < nsplits && ok; s += a.npairs) {
            const MlaSplit sp = split_info(ln, chunk, s);
            for (int p = sp.p0; p < sp.p1; ++p, ++g) {
                const int sbuf = g % kStages;
                if (aborted() || !wait_all(B(s_full + sbuf), (g / kStages) & 1, a.status) ||
                    (g >= 1 && !wait_all_cluster(B(peer_free), (g - 1) & 1, a.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t src = tmem + tl + TM_S + sbuf * kTok;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(src + h2 * 32, v);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_async_v4(peer_row + (h2 * 8 + c) * 2048, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3],
                                    peer_recv_full);
                }
                tc_fence_before();
                mbar_arrive(B(s_read + sbuf));
            }
        }
        if (!ok && lane == 0) abort_pair();
    } else {
        // ---------------------------------------------------------------- softmax, epilogue
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;                 // head = TMEM lane
        const uint32_t tl = (uint32_t)(q4 * 32) << 16;
        const int st_tid = threadIdx.x - 96;            // 0..127
        // Receive buffer [16 chunks][128 rows][16 B]: chunk c of every row is contiguous, so one
        // warp's store of a chunk is a single 512-byte write from the peer, and its load here
        // touches 32 consecutive 16-byte words.
        const uint32_t peer_peer_free = peer_addr(B(peer_free), peer);
        bool ok = true;
        int g = 0;
        if (st_tid == 0) mbar_arrive_expect_tx(B(recv_full), 128 * 256);  // receive phase of tile 0
        for (int s = pair; s < nsplits && ok; s += a.npairs) {
            const MlaSplit sp = split_info(ln, chunk, s);
            const int L = sp.b < kSeqCache ? reinterpret_cast<const int*>(smem + OFF_SEQ)[sp.b] : a.seq_lens[sp.b];
            float mref = -INFINITY, l = 0.f;
            for (int p = sp.p0; p < sp.p1; ++p, ++g) {
                const int st = g % kStages;
                if (aborted() || !wait_all(B(s_full + st), (g / kStages) & 1, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // own partial of tile g, plus the peer's from the receive buffer
                const uint32_t sb = tmem + tl + TM_S + st * kTok;
                uint32_t sv[kTok];
                tmem_ld_32x32b_x32_nowait(sb, sv);
                tmem_ld_32x32b_x32_nowait(sb + 32, sv + 32);
                if (!wait_all_cluster(B(recv_full), g & 1, a.status)) {
                    ok = false;
                    break;
                }
                tmem_wait_ld();
                const float4* rr = reinterpret_cast<const float4*>(smem + OFF_RECV + row * 16);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 w = rr[c * 128];
                    sv[4 * c] = __float_as_uint(__uint_as_float(sv[4 * c]) + w.x);
                    sv[4 * c + 1] = __float_as_uint(__uint_as_float(sv[4 * c + 1]) + w.y);
                    sv[4 * c + 2] = __float_as_uint(__uint_as_float(sv[4 * c + 2]) + w.z);
                    sv[4 * c + 3] = __float_as_uint(__uint_as_float(sv[4 * c + 3]) + w.w);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_remote_relaxed(peer_peer_free);
                if (st_tid == 0) mbar_arrive_expect_tx(B(recv_full), 128 * 256);  // receive phase of tile g+1
                // Tokens past the sequence end: -inf logits, and their value rows cleared (the
                // pool may hold any bits there) before P.V reads them.
                const int nvalid = min(kTok, L - p * kTok);
                if (nvalid < kTok) {
                    // the page's copy has landed (its score MMA ran); waiting on it orders these
                    // stores after the copy's writes
                    if (!wait_all(B(k_full + st), (g / kStages) & 1, a.status)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int e = 0; e < kTok; ++e) sv[e] = e < nvalid ? sv[e] : 0xff800000u;
                    const int t = st_tid & 63;
                    if (t >= nvalid) {
                        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            uint4* dst = reinterpret_cast<uint4*>(smem + OFF_KV + st * STAGE +
                                                                  ((st_tid >> 6) * 2 + h2) * KATOM + t * 128);
#pragma unroll
                            for (int i = 0; i < 8; ++i) dst[i] = z;
                        }
                    }
                }
                float m8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmaxf(__uint_as_float(sv[i]), __uint_as_float(sv[8 + i]));
#pragma unroll
                for (int e = 16; e < kTok; e += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        m8[i] = fmax3(m8[i], __uint_as_float(sv[e + i]), __uint_as_float(sv[e + 8 + i]));
                float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                mx *= a.scale_log2;
                const float mnew = fmaxf(mref, mx);
                const bool raise = mnew > mref + kRescaleThreshold;
                const float muse = raise ? mnew : mref;
                const float alpha = raise ? ((mref == -INFINITY) ? 0.f : ex2_approx(mref - mnew)) : 1.f;
                const float nm = muse == -INFINITY ? -INFINITY : -muse;
                float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = ex2_approx(fmaf(__uint_as_float(sv[hh * 32 + e]), a.scale_log2, nm));
                        const float p1 = ex2_approx(fmaf(__uint_as_float(sv[hh * 32 + e + 1]), a.scale_log2, nm));
                        r8[(e >> 1) & 7] += p0 + p1;
                        pk[e / 2] = pack_bf16x2(p0, p1);
                    }
                    tmem_st_32x32b_x16(sb + hh * 16, pk);
                }
                const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
                l = l * alpha + rs;
                mref = muse;
                // O is rescaled (after the previous P.V has finished accumulating) only when a row's
                // max rose by more than 2^8; otherwise this tile's P.V queues behind the last one.
                if (p > sp.p0 && __any_sync(0xffffffffu, raise)) {
                    if (!wait_all(B(o_done + (g - 1) % kStages), ((g - 1) / kStages) & 1, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t v[32];
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        tmem_ld_32x32b_x32(tmem + tl + TM_O + c * 32, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st_32x32b_x32(tmem + tl + TM_O + c * 32, v);
                    }
                }
                tmem_wait_st();
                if (nvalid < kTok) fence_proxy_async_smem();  // cleared value rows before the tensor core reads them
                tc_fence_before();
                mbar_arrive(B(p_full));
            }
            if (!ok) break;
            // ---- split epilogue: (m, l) and this CTA's 256 columns of the unnormalised O
            if (!wait_all(B(o_done + (g - 1) % kStages), ((g - 1) / kStages) & 1, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (row < a.H) {
                if (rank == 0)
                    *reinterpret_cast<float2*>(a.part_ml + ((size_t)row * a.pmax + s) * 2) = make_float2(mref, l);
            }
            float* dst = a.part_acc + ((size_t)row * a.pmax + s) * kDC + col0;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + tl + TM_O + c * 32, v);
                if (row < a.H) {
                    float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                            __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
            tc_fence_before();  // O read before the next split's first P.V overwrites it
        }
        if (!ok) {
            if (lane == 0) abort_pair();
            // Asynchronous stores the peer issued into this CTA's receive buffer may still be in
            // flight when a wait gave up; give them time to land before the CTA can exit.
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 20000) __nanosleep(1000);
        }
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
    // No CTA leaves while its peer may still write into its shared memory.
    cluster_sync_all();
}

// Log-sum-exp merge of a sequence's split partials per head, bf16 out.  grid (H, B), 256 threads
// (two latent columns each); the split weights 2^(m_i - M) are formed once per block.
// A sequence has at most max(npairs, 1) splits (the partition gives every sequence one split once
// B >= npairs), far below this on any GPU the host sizes npairs for.
constexpr int kMaxCombine = 256;
__global__ void __launch_bounds__(256) mla_combine_kernel(const MlaArgs a) {
    pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y;
    const int first = a.seq_first[b], count = a.seq_count[b];
    const int c = threadIdx.x * 2;
    uint32_t* o = reinterpret_cast<uint32_t*>(a.out + ((size_t)b * a.H + h) * kDC + c);
    if (count == 0 || count > kMaxCombine) {
        if (h == 0 && threadIdx.x == 0) set_status(a.status, LRKV_DEV_BAD_SEQLEN);
        *o = 0u;
        return;
    }
    const float* ml = a.part_ml + ((size_t)h * a.pmax + first) * 2;
    __shared__ float wsh[kMaxCombine];
    __shared__ float lsh;
    const int cs = count;
    if (threadIdx.x < 32) {
        float M = -INFINITY;
        for (int i = threadIdx.x; i < count; i += 32) M = fmaxf(M, ml[2 * i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float Ls = 0.f;
        for (int i = threadIdx.x; i < count; i += 32) {
            const float w = exp2f(ml[2 * i] - M);
            wsh[i] = w;
            Ls = fmaf(w, ml[2 * i + 1], Ls);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
        if (threadIdx.x == 0) lsh = Ls;
    }
    __syncthreads();
    const float* acc = a.part_acc + ((size_t)h * a.pmax + first) * kDC + c;
    float v0 = 0.f, v1 = 0.f;
    int i = 0;
    // four partial rows in flight at a time
    for (; i + 4 <= cs; i += 4) {
        const float2 x0 = *reinterpret_cast<const float2*>(acc + (size_t)(i + 0) * kDC);
        const float2 x1 = *reinterpret_cast<const float2*>(acc + (size_t)(i + 1) * kDC);
        const float2 x2 = *reinterpret_cast<const float2*>(acc + (size_t)(i + 2) * kDC);
        const float2 x3 = *reinterpret_cast<const float2*>(acc + (size_t)(i + 3) * kDC);
        v0 = fmaf(wsh[i], x0.x, v0);
        v1 = fmaf(wsh[i], x0.y, v1);
        v0 = fmaf(wsh[i + 1], x1.x, v0);
        v1 = fmaf(wsh[i + 1], x1.y, v1);
        v0 = fmaf(wsh[i + 2], x2.x, v0);
        v1 = fmaf(wsh[i + 2], x2.y, v1);
        v0 = fmaf(wsh[i + 3], x3.x, v0);
        v1 = fmaf(wsh[i + 3], x3.y, v1);
    }
    for (; i < cs; ++i) {
        const float2 x = *reinterpret_cast<const float2*>(acc + (size_t)i * kDC);
        v0 = fmaf(wsh[i], x.x, v0);
        v1 = fmaf(wsh[i], x.y, v1);
    }
    const float inv = lsh > 0.f ? 1.f / lsh : 0.f;
    *o = pack_bf16x2(v0 * inv, v1 * inv);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t mla_workspace_bytes(int H, int B, int npairs) {
    const size_t pmax = (size_t)max(npairs, B);
    return align256(pmax * H * 2 * sizeof(float)) + align256(pmax * H * kDC * sizeof(float)) +
           2 * align256((size_t)B * sizeof(int));
}

void mla_carve_workspace(MlaArgs* a, void* ws) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    a->part_ml = reinterpret_cast<float*>(base);
    base += align256((size_t)a->pmax * a->H * 2 * sizeof(float));
    a->part_acc = reinterpret_cast<float*>(base);
    base += align256((size_t)a->pmax * a->H * kDC * sizeof(float));
    a->seq_first = reinterpret_cast<int*>(base);
    base += align256((size_t)a->B * sizeof(int));
    a->seq_count = reinterpret_cast<int*>(base);
}

cudaError_t launch_mla_decode(const CUtensorMap& tmQ, const CUtensorMap& tmQr, const CUtensorMap& tmKV,
                              const CUtensorMap& tmKVr, const MlaArgs& a, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    // An ordinary launch: the split must not start reading the cache before the caller's previous
    // kernel on the stream (an append of the newest rows) has finished.
    mla_decode_split_kernel<<<2 * a.npairs, kThreads, kSmemBytes, stream>>>(tmQ, tmQr, tmKV, tmKVr, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.H, a.B);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_combine_kernel, a);
}

}  // namespace lrkv
