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
// that divide the columns: rank 0 owns c[0:256), rank 1 owns c[256:512) and k^R.  Each
// CTA loads only its columns of Q and of every page (every cached byte is read once),
// computes the partial logits S_r = Q_r K_r^T, and the two exchange S_r through
// distributed shared memory; both then hold S = S_0 + S_1 (fp32 addition commutes, so the
// two softmaxes agree bit for bit) and each accumulates its own half O_r += P V_r, with
// V_r = its 256 latent columns of the same page.  Splits write (m, l, O) partials; a
// combine kernel merges them per (sequence, head) by log-sum-exp.
//
// Warp roles per CTA: warp 0 TMA producer (Q per split, 2-stage page ring), warp 1 score
// MMAs and TMEM owner, warp 2 P.V MMAs, warps 3-6 softmax and exchange (one head row per
// thread, TMEM lane quarter = warp % 4).  Every wait is bounded; an expired wait sets
// LRKV_DEV_TIMEOUT and the abort flag of both CTAs of the pair.
#include <type_traits>

#include "kernels.h"
#include "lrkv_internal.cuh"
#include "mla.h"

namespace lrkv {

namespace {

constexpr int kDC = 512, kDR = 64, kDK = kDC + kDR;
constexpr int kTok = 64;                        // tokens per tile (one page)
constexpr int kMaxAtoms = 5;                    // 64-column blocks per CTA: rank 0 four, rank 1 five
constexpr uint32_t QATOM = 128 * 128;           // [128 heads][64 columns] bf16, 128-byte swizzle
constexpr uint32_t KATOM = kTok * 128;          // [64 tokens][64 columns] bf16, 128-byte swizzle
constexpr int kStages = 2;
constexpr uint32_t STAGE = kMaxAtoms * KATOM;   // 40 KiB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = kMaxAtoms * QATOM;                // 80 KiB
constexpr uint32_t OFF_RECV = OFF_KV + kStages * STAGE;      // [128][64] fp32 partial logits from the peer
constexpr uint32_t OFF_BAR = OFF_RECV + 128 * 256;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;
constexpr uint32_t TM_S0 = 0, TM_S1 = 64, TM_O = 128, TM_COLS = 512;
constexpr int kThreads = 224;
constexpr float kRescaleThreshold = 8.0f;      // log2 units

static_assert(kDK == 576, "row width");
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
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's prior writes.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
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
__device__ __forceinline__ uint64_t vdesc(uint32_t a) { return sdesc(a, KATOM, 1024, 2); }

// ---- partition: a sequence's pages are cut into contiguous splits of about equal size,
// at most max(npairs, B) splits in all (every split lies inside one sequence).
struct MlaSplit {
    int b, p0, p1;
};

__device__ __forceinline__ int seq_pages(const MlaArgs& a, int b) {
    const int L = a.seq_lens[b];
    return (L >= 1 && L <= a.max_pages * kTok) ? (L + kTok - 1) / kTok : 0;
}

__device__ __forceinline__ int partition_chunk(const MlaArgs& a, int* nsplits) {
    long long total = 0;
    for (int b = 0; b < a.B; ++b) total += seq_pages(a, b);
    const int G = a.npairs;
    const int denom = G > a.B ? G - a.B : 1;
    const int chunk = (int)max(1LL, (total + denom - 1) / denom);
    int ns = 0;
    for (int b = 0; b < a.B; ++b) ns += (seq_pages(a, b) + chunk - 1) / chunk;
    *nsplits = ns;
    return chunk;
}

__device__ __forceinline__ MlaSplit split_info(const MlaArgs& a, int chunk, int s) {
    int base = 0;
    for (int b = 0; b < a.B; ++b) {
        const int gr = seq_pages(a, b);
        const int ns = (gr + chunk - 1) / chunk;
        if (s < base + ns) {
            const int i = s - base;
            return MlaSplit{b, (int)((long long)i * gr / ns), (int)((long long)(i + 1) * gr / ns)};
        }
        base += ns;
    }
    return MlaSplit{0, 0, 0};
}

__device__ __forceinline__ void seq_splits(const MlaArgs& a, int chunk, int b, int* first, int* count) {
    int base = 0;
    for (int bb = 0; bb < b; ++bb) base += (seq_pages(a, bb) + chunk - 1) / chunk;
    *first = base;
    *count = (seq_pages(a, b) + chunk - 1) / chunk;
}

// Score MMAs of one CTA: S_r = Q_r . K_r^T over its NA column blocks (NA * 4 K-steps of 16).
// The tile loop branches on the ring stage so that every descriptor is loop-invariant.
template <int NA>
__device__ __forceinline__ bool score_mmas(const MlaArgs& a, uint32_t S0, uint32_t tmem, uint64_t* bars,
                                           volatile int* abort_flag, int pair, int nsplits, int chunk) {
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* k_full = bars + 2;
    uint64_t* s_full = bars + 6;
    uint64_t* s_free = bars + 8;
    auto B = [&](uint64_t* p) { return smem_u32(p); };
    constexpr uint32_t id_S = idesc_bf16_f32(128, kTok);
    const uint64_t dQ = kdesc(S0 + OFF_Q), dK = kdesc(S0 + OFF_KV);
    auto kq = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * QATOM + (kk & 3) * 32) >> 4); };
    auto kk_ = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * KATOM + (kk & 3) * 32) >> 4); };
    auto tile = [&](int g, auto ST) -> bool {
        constexpr int st = decltype(ST)::value;
        if (__any_sync(0xffffffffu, *abort_flag != 0) || !wait_all(B(k_full + st), (g >> 1) & 1, a.status) ||
            (g >= 2 && !wait_all(B(s_free + st), ((g >> 1) - 1) & 1, a.status)))
            return false;
        tc_fence_after();
        constexpr uint64_t so = (uint64_t)(st * STAGE) >> 4;
        const uint32_t d = tmem + (st ? TM_S1 : TM_S0);
#pragma unroll
        for (int kk = 0; kk < NA * 4; ++kk)
            if (elect_one_sync()) tc_mma_bf16(d, dQ + kq(kk), dK + so + kk_(kk), id_S, kk > 0);
        if (elect_one_sync()) tc_commit(B(s_full + st));
        __syncwarp();
        return true;
    };
    bool ok = true;
    int g = 0, sidx = 0;
    for (int s = pair; s < nsplits && ok; s += a.npairs, ++sidx) {
        const MlaSplit sp = split_info(a, chunk, s);
        ok = wait_all(B(q_full), sidx & 1, a.status);
        if (ok) tc_fence_after();
        for (int p = sp.p0; p < sp.p1 && ok; ++p, ++g)
            ok = (g & 1) ? tile(g, std::integral_constant<int, 1>{}) : tile(g, std::integral_constant<int, 0>{});
        // Q may be replaced once every score MMA of this split has read it
        if (elect_one_sync()) tc_commit(B(q_empty));
        __syncwarp();
    }
    return ok;
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_split_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                            const MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzle atoms; the offset is the same in both CTAs of the
    // pair (same kernel, same dynamic shared-memory base), so mapped addresses line up.
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t S0 = smem_u32(smem);
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int na = rank ? 5 : 4;   // column blocks of this CTA
    const int col0 = rank * 256;   // first cache column of this CTA
    const int pair = blockIdx.x >> 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* q_full = bars + 0;     // Q of the split landed
    uint64_t* q_empty = bars + 1;    // score MMAs of the split done with Q
    uint64_t* k_full = bars + 2;     // [2] page landed
    uint64_t* k_empty = bars + 4;    // [2] P.V done with the page
    uint64_t* s_full = bars + 6;     // [2] partial S in TMEM
    uint64_t* s_free = bars + 8;     // [2] P.V done with the P held in that S buffer
    uint64_t* p_full = bars + 10;    // softmax wrote P (128 arrivals)
    uint64_t* o_done = bars + 11;    // [2] P.V of the tile (by parity) complete
    uint64_t* recv_full = bars + 13; // the peer's partial S is in this CTA's receive buffer (128 remote arrivals)
    uint64_t* peer_free = bars + 14; // the peer has read what this CTA wrote into its buffer (128 remote arrivals)
    uint64_t* mma_drain = bars + 15;
    uint64_t* pv_drain = bars + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
    volatile int* abort_flag = reinterpret_cast<int*>(bars + 18);
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(B(k_full + i), 1);
            mbar_init(B(k_empty + i), 1);
            mbar_init(B(s_full + i), 1);
            mbar_init(B(s_free + i), 1);
            mbar_init(B(o_done + i), 1);
        }
        mbar_init(B(p_full), 128);
        mbar_init(B(recv_full), 128);
        mbar_init(B(peer_free), 128);
        mbar_init(B(mma_drain), 1);
        mbar_init(B(pv_drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int nsplits;
    const int chunk = partition_chunk(a, &nsplits);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        const uint64_t pol = policy_evict_first();
        bool ok = true;
        int g = 0, sidx = 0, q_issued = -1;
        for (int s = pair; s < nsplits && ok; s += a.npairs, ++sidx) {
            const MlaSplit sp = split_info(a, chunk, s);
            if ((sidx > 0 && !wait_all(B(q_empty), (sidx - 1) & 1, a.status)) || aborted()) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(B(q_full), na * QATOM);
                for (int i = 0; i < na; ++i)
                    tma_load_3d(S0 + OFF_Q + i * QATOM, &tmQ, col0 + i * 64, 0, sp.b, B(q_full));
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
            for (int j = 0; j < sp.p1 - sp.p0; ++j, ++g) {
                if (j > 0 && (j & 31) == 0) {
                    cur = nxt;
                    nxt = fetch((j >> 5) + 1);
                }
                const int row = __shfl_sync(0xffffffffu, cur, j & 31);
                const int st = g & 1;
                if ((g >= 2 && !wait_all(B(k_empty + st), ((g >> 1) - 1) & 1, a.status)) || aborted()) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t dst = S0 + OFF_KV + st * STAGE, bar = B(k_full + st);
                    mbar_arrive_expect_tx(bar, na * KATOM);
                    for (int i = 0; i < na; ++i) tma_load_2d_hint(dst + i * KATOM, &tmKV, col0 + i * 64, row, bar, pol);
                }
                __syncwarp();
            }
        }
        if (!ok) {
            if (lane == 0) abort_pair();
            // let the copies still in flight land before the CTA exits
            for (int k = max(0, g - 2); k < g; ++k) wait_all(B(k_full + (k & 1)), (k >> 1) & 1, a.status);
            if (q_issued >= 0) wait_all(B(q_full), q_issued & 1, a.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- score MMAs
        const bool ok = rank ? score_mmas<5>(a, S0, tmem, bars, abort_flag, pair, nsplits, chunk)
                             : score_mmas<4>(a, S0, tmem, bars, abort_flag, pair, nsplits, chunk);
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
        auto pv = [&](int g, bool first, auto ST) -> bool {
            constexpr int st = decltype(ST)::value;
            if (aborted() || !wait_all(B(p_full), g & 1, a.status)) return false;
            tc_fence_after();
            constexpr uint64_t so = (uint64_t)(st * STAGE) >> 4;
            const uint32_t pt = tmem + (st ? TM_S1 : TM_S0);
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
            const MlaSplit sp = split_info(a, chunk, s);
            for (int p = sp.p0; p < sp.p1 && ok; ++p, ++g) {
                const bool first = p == sp.p0;
                ok = (g & 1) ? pv(g, first, std::integral_constant<int, 1>{})
                             : pv(g, first, std::integral_constant<int, 0>{});
            }
        }
        if (!ok && lane == 0) abort_pair();
        if (elect_one_sync()) tc_commit(B(pv_drain));
        __syncwarp();
        wait_all(B(pv_drain), 0, a.status);
    } else {
        // ---------------------------------------------------------------- softmax, exchange, epilogue
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;                 // head = TMEM lane
        const uint32_t tl = (uint32_t)(q4 * 32) << 16;
        const int st_tid = threadIdx.x - 96;            // 0..127
        const uint32_t recv_row = S0 + OFF_RECV + row * 256;
        const uint32_t peer_row = peer_addr(recv_row, peer);
        const uint32_t peer_recv_full = peer_addr(B(recv_full), peer);
        const uint32_t peer_peer_free = peer_addr(B(peer_free), peer);
        const int sw = row & 15;                        // 16-byte chunk swizzle of the receive rows
        bool ok = true;
        int g = 0;
        for (int s = pair; s < nsplits && ok; s += a.npairs) {
            const MlaSplit sp = split_info(a, chunk, s);
            const int L = a.seq_lens[sp.b];
            float mref = -INFINITY, l = 0.f;
            for (int p = sp.p0; p < sp.p1; ++p, ++g) {
                const int st = g & 1;
                if (aborted() || !wait_all(B(s_full + st), (g >> 1) & 1, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sb = tmem + tl + (st ? TM_S1 : TM_S0);
                uint32_t sv[kTok];
                tmem_ld_32x32b_x32_nowait(sb, sv);
                tmem_ld_32x32b_x32_nowait(sb + 32, sv + 32);
                tmem_wait_ld();
                // Exchange the partial logits: ours into the peer's receive buffer (once the peer
                // has read the previous tile from it), then theirs out of ours.
                if (g >= 1 && !wait_all_cluster(B(peer_free), (g - 1) & 1, a.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    st_cluster_v4(peer_row + ((c ^ sw) << 4), sv[4 * c], sv[4 * c + 1], sv[4 * c + 2], sv[4 * c + 3]);
                mbar_arrive_remote(peer_recv_full);
                if (!wait_all_cluster(B(recv_full), g & 1, a.status)) {
                    ok = false;
                    break;
                }
                const float4* rr = reinterpret_cast<const float4*>(smem + OFF_RECV + row * 256);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 w = rr[c ^ sw];
                    sv[4 * c] = __float_as_uint(__uint_as_float(sv[4 * c]) + w.x);
                    sv[4 * c + 1] = __float_as_uint(__uint_as_float(sv[4 * c + 1]) + w.y);
                    sv[4 * c + 2] = __float_as_uint(__uint_as_float(sv[4 * c + 2]) + w.z);
                    sv[4 * c + 3] = __float_as_uint(__uint_as_float(sv[4 * c + 3]) + w.w);
                }
                mbar_arrive_remote(peer_peer_free);
                // Tokens past the sequence end: -inf logits, and their value rows cleared (the
                // pool may hold any bits there) before P.V reads them.
                const int nvalid = min(kTok, L - p * kTok);
                if (nvalid < kTok) {
                    // the page's copy has landed (its score MMA ran); waiting on it orders these
                    // stores after the copy's writes
                    if (!wait_all(B(k_full + st), (g >> 1) & 1, a.status)) {
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
                uint32_t pk[kTok / 2];
#pragma unroll
                for (int e = 0; e < kTok; e += 2) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), a.scale_log2, nm));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), a.scale_log2, nm));
                    r8[(e >> 1) & 7] += p0 + p1;
                    pk[e / 2] = pack_bf16x2(p0, p1);
                }
                tmem_st_32x32b_x32(sb, pk);
                const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
                l = l * alpha + rs;
                mref = muse;
                // O is rescaled (after the previous P.V has finished accumulating) only when a row's
                // max rose by more than 2^8; otherwise this tile's P.V queues behind the last one.
                if (p > sp.p0 && __any_sync(0xffffffffu, raise)) {
                    if (!wait_all(B(o_done + ((g - 1) & 1)), ((g - 1) >> 1) & 1, a.status)) {
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
                fence_proxy_async_smem();  // cleared value rows (if any) before the tensor core reads them
                tc_fence_before();
                mbar_arrive(B(p_full));
            }
            if (!ok) break;
            // ---- split epilogue: (m, l) and this CTA's 256 columns of the unnormalised O
            if (!wait_all(B(o_done + ((g - 1) & 1)), ((g - 1) >> 1) & 1, a.status)) {
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
        if (!ok && lane == 0) abort_pair();
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
// (two latent columns each).
__global__ void __launch_bounds__(256) mla_combine_kernel(const MlaArgs a) {
    pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y;
    int nsplits;
    const int chunk = partition_chunk(a, &nsplits);
    int first, count;
    seq_splits(a, chunk, b, &first, &count);
    const int c = threadIdx.x * 2;
    uint32_t* o = reinterpret_cast<uint32_t*>(a.out + ((size_t)b * a.H + h) * kDC + c);
    if (count == 0) {
        if (h == 0 && threadIdx.x == 0) set_status(a.status, LRKV_DEV_BAD_SEQLEN);
        *o = 0u;
        return;
    }
    const float* ml = a.part_ml + ((size_t)h * a.pmax + first) * 2;
    float M = -INFINITY;
    for (int i = 0; i < count; ++i) M = fmaxf(M, ml[2 * i]);
    float Ls = 0.f, v0 = 0.f, v1 = 0.f;
    const float* acc = a.part_acc + ((size_t)h * a.pmax + first) * kDC + c;
    for (int i = 0; i < count; ++i) {
        const float w = exp2f(ml[2 * i] - M);
        Ls = fmaf(w, ml[2 * i + 1], Ls);
        const float2 x = *reinterpret_cast<const float2*>(acc + (size_t)i * kDC);
        v0 = fmaf(w, x.x, v0);
        v1 = fmaf(w, x.y, v1);
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    *o = pack_bf16x2(v0 * inv, v1 * inv);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t mla_workspace_bytes(int H, int B, int npairs) {
    const size_t pmax = (size_t)max(npairs, B);
    return align256(pmax * H * 2 * sizeof(float)) + align256(pmax * H * kDC * sizeof(float));
}

void mla_carve_workspace(MlaArgs* a, void* ws) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    a->part_ml = reinterpret_cast<float*>(base);
    base += align256((size_t)a->pmax * a->H * 2 * sizeof(float));
    a->part_acc = reinterpret_cast<float*>(base);
}

cudaError_t launch_mla_decode(const CUtensorMap& tmQ, const CUtensorMap& tmKV, const MlaArgs& a,
                              cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    // An ordinary launch: the split must not start reading the cache before the caller's previous
    // kernel on the stream (an append of the newest rows) has finished.
    mla_decode_split_kernel<<<2 * a.npairs, kThreads, kSmemBytes, stream>>>(tmQ, tmKV, a);
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
