// decode_work.cuh -- the work plan of the decode's split-K scan, shared by the CUDA-core
// and the tensor-core scan kernels: how a call's cached tokens are cut into pieces of
// work, one per SM, and how a CTA walks its segments.
#pragma once

#include "kernels.h"
#include "lrkv_internal.cuh"

namespace lrkv {

constexpr int kGran = 8;                              // tokens per pipeline stage (granule)
constexpr int kScratchFloats = 16 * 8 + 16 * 8 + 16;  // per consumer warp: z-scores, p, alpha
constexpr int kPageCache = 64;                        // page ids of a segment kept in shared memory

constexpr int kSeqCache = 128;                        // sequence lengths kept in shared memory
constexpr int kMaxGroups = 8;                         // consumer groups at most (8 warps, one per group)

// Row stride (floats) of a head's accumulator in the shared-memory staging of the group merge:
// W itself when W = 8 or 24 (mod 32), else W + 8, so that the rows of one MMA fragment (8
// heads) start 8 or 24 banks apart.
__host__ __device__ constexpr int decode_stage_stride(int W) { return (W % 16 == 0) ? W + 8 : W; }

// The work of a decode call: nvb = layers * B virtual sequences vb = layer * B + b (all
// layers share the block table and lengths), each cut into 8-token granules, T granules in
// all, scanned by `nranges` CTA-sized pieces of work.  With head groups every (layer,
// sequence) pair appears as `groups` consecutive virtual sequences, one per group of heads
// (Work::B then counts groups x sequences per layer).  Two ways to cut, chosen identically by
// every CTA (plan()):
//  - pieces: every sequence is cut into ceil(gr / chunk) near-equal pieces, with the smallest
//    chunk for which all pieces number at most nranges; each piece is one segment with its
//    own partial slot (the piece's global index).  No CTA crosses a sequence boundary, so no
//    pipeline drains between sequences; used when the largest piece costs at most a pipeline
//    drain-and-refill (`bubble` granules) more than an exact split would.
//  - ranges: the granules of all virtual sequences, concatenated in vb order, are divided
//    into nranges contiguous ranges of equal size (+-1): range c is [floor(c T / nranges),
//    floor((c + 1) T / nranges)) (nranges first clamped to T, so that no range is empty).  A
//    range covers one or more segments of consecutive sequences; the segment of sequence vb
//    inside range c writes partial slot vb + c, so each sequence's partials sit in
//    consecutive slots.  Used when the sequences are too many or too uneven for pieces.
// Either way the slots number at most nvb + nranges.
// All counts are 32-bit (the host bounds T below 2^31 and nranges by 2^16): one thread
// computes the plan before the first load of the CTA is issued, and a 64-bit division is a
// long dependent software sequence on the GPU.  floor(c T / n) is formed as c (T / n) +
// floor(c (T mod n) / n), whose product c (T mod n) < n^2 fits in 32 unsigned bits.
struct Work {
    const int32_t* g;  // lengths in global memory
    const int* s;      // shared-memory copy of the first kSeqCache
    int B, layers, cap, nranges;
    int Tb;            // granules of one layer (all B sequences)
    int pieces;        // 1: pieces, 0: ranges
    int chunk;         // pieces: largest piece, in granules
    int per_layer_pieces;
    int rq, rr;        // ranges: T / nranges and T mod nranges
    int lgh;           // log2 of the head groups: entry b of a layer is sequence b >> lgh

    __device__ __forceinline__ int len(int b) const {
        const int q = b >> lgh;
        return q < kSeqCache ? s[q] : g[q];
    }
    // Granules of sequence b, or 0 when its length is outside [1, cap].
    __device__ __forceinline__ int gran_b(int b) const {
        const int L = len(b);
        return (L >= 1 && L <= cap) ? (L + kGran - 1) / kGran : 0;
    }
    __device__ __forceinline__ int gran(int vb) const { return gran_b(vb % B); }
    __device__ __forceinline__ int total() const { return Tb * layers; }
    __device__ __forceinline__ int range_start(int c) const {
        return c * rq + (int)(((unsigned)c * (unsigned)rr) / (unsigned)nranges);
    }
    // Index of the range that holds granule gi (0 <= gi < total()): a float estimate of
    // floor(gi nranges / T), off by at most one, stepped to the range whose bounds hold gi.
    __device__ __forceinline__ int range_of(int gi) const {
        int c = (int)((float)gi * (float)nranges / (float)total());
        c = min(max(c, 0), nranges - 1);
        while (c + 1 < nranges && range_start(c + 1) <= gi) ++c;
        while (c > 0 && range_start(c) > gi) --c;
        return c;
    }
    // The (non-empty) virtual sequence that holds granule gi, and its first granule.
    __device__ __forceinline__ void locate(int gi, int* vb, int* start) const {
        const int l = (int)((unsigned)gi / (unsigned)Tb);
        int p = Tb * l;
        int b = 0;
        while (b < B - 1 && p + gran_b(b) <= gi) p += gran_b(b++);
        *vb = l * B + b;
        *start = p;
    }
    // Pieces of sequence b with largest piece c.
    __device__ __forceinline__ int npieces(int b, int c) const {
        return (int)((unsigned)(gran_b(b) + c - 1) / (unsigned)c);
    }
    // Pieces mode: virtual sequence and granule range of piece pc.
    __device__ __forceinline__ void piece(int pc, int* vb, int* g0, int* g1) const {
        const int l = (int)((unsigned)pc / (unsigned)per_layer_pieces);
        int base = per_layer_pieces * l;
        int b = 0;
        for (;; ++b) {
            const int n = npieces(b, chunk);
            if (pc < base + n || b == B - 1) break;
            base += n;
        }
        const unsigned gr = (unsigned)gran_b(b);
        const unsigned np = (gr + chunk - 1) / (unsigned)chunk;
        const unsigned i = (unsigned)(pc - base);
        // floor(i gr / np) with i < np <= 2^16
        const unsigned q = gr / np, r = gr - q * np;
        *vb = l * B + b;
        *g0 = (int)(i * q + (i * r) / np);
        *g1 = (int)((i + 1) * q + ((i + 1) * r) / np);
    }

    // Sum (max for gmax) over the NL lanes that share a plan (a no-op for one thread).
    template <int NL>
    __device__ __forceinline__ static int lanes_sum(int v) {
        if (NL > 1) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        }
        return v;
    }
    // Counts the granules and chooses the cut.  NL = 1: one thread alone walks every sequence
    // (cheap for small batches, and needs no barrier when every thread does it); NL = 32: a full
    // warp, lanes taking every 32nd sequence, sums exchanged by shuffles (every lane ends with
    // the same plan; publish() then hands it to the rest of the block).
    template <int NL>
    __device__ __forceinline__ void plan(int bubble, int lane) {
        int tb = 0, nonempty = 0, gmax = 0;
        for (int b = lane; b < B; b += NL) {
            const int gr = gran_b(b);
            tb += gr;
            nonempty += gr > 0;
            gmax = max(gmax, gr);
        }
        tb = lanes_sum<NL>(tb);
        nonempty = lanes_sum<NL>(nonempty);
        if (NL > 1) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) gmax = max(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
        }
        Tb = tb;
        const unsigned T = (unsigned)total();
        if ((int)T < nranges) nranges = (int)T;  // no empty range
        pieces = 0;
        rq = nranges > 0 ? (int)(T / (unsigned)nranges) : 0;
        rr = nranges > 0 ? (int)(T - (unsigned)rq * (unsigned)nranges) : 0;
        const int occupied = nonempty * layers;
        if (T == 0 || occupied > nranges) return;
        // Two candidate piece sizes: the exact share ceil(T / nranges), when its pieces fit in
        // nranges, else c0 = ceil(T / (nranges - occupied)), which always fits (sum ceil(gr / c0)
        // <= T / c0 + occupied).  (A search between them gained nothing measurable and, code
        // being what it is, its loop made the stage loop slower.)
        const int share = rq + (rr != 0);
        const int c0 = occupied < nranges
                           ? (int)((T + (unsigned)(nranges - occupied) - 1) / (unsigned)(nranges - occupied))
                           : gmax;
        int c = min(share, gmax);
        int n = 0;
        for (int b = lane; b < B; b += NL) n += npieces(b, c);
        n = lanes_sum<NL>(n);
        if (n * layers > nranges) {
            c = min(c0, gmax);
            n = 0;
            for (int b = lane; b < B; b += NL) n += npieces(b, c);
            n = lanes_sum<NL>(n);
        }
        if (c <= share + bubble) {
            pieces = 1;
            chunk = c;
            per_layer_pieces = n;
        }
    }
    // Number of pieces of work (CTA iterations) of the call.
    __device__ __forceinline__ int work_items() const { return pieces ? per_layer_pieces * layers : nranges; }
};

// This CTA's walk over its segments: (virtual sequence, granule range in it, partial slot).
struct SegWalk {
    int item;            // current piece or range
    int gcur, gend, vstart;
    int seg_start;       // ranges: first granule (in the concatenation) of the last segment returned
    int vb;

    __device__ __forceinline__ void start(int first_item) {
        item = first_item;
        gcur = gend = 0;
        vb = 0;
        vstart = 0;
    }
    __device__ __forceinline__ bool next(const Work& w, int* vb_out, int* g0, int* g1, int* slot) {
        if (w.pieces) {
            if (item >= w.work_items()) return false;
            w.piece(item, vb_out, g0, g1);
            *slot = item;
            item += gridDim.x;
            return true;
        }
        const int nvb = w.layers * w.B;
        if (gcur >= gend) {
            if (gend > 0) item += gridDim.x;  // the current range is done
            if (item >= w.nranges) return false;
            gcur = w.range_start(item);
            gend = w.range_start(item + 1);
            w.locate(gcur, &vb, &vstart);
        }
        const int gr = w.gran(vb);
        const int se = min(gend, vstart + gr);
        *vb_out = vb;
        *g0 = gcur - vstart;
        *g1 = se - vstart;
        *slot = vb + item;
        seg_start = gcur;
        gcur = se;
        if (gcur == vstart + gr) {
            vstart += gr;
            do {
                ++vb;
            } while (vb < nvb && w.gran(vb) == 0);
        }
        return true;
    }
};

// The split kernel's control block in shared memory: the plan and this CTA's walk over its
// segments, advanced by thread 0 at each segment boundary and read by all threads after a
// barrier (kept out of the registers that the stage loop needs).
struct SplitCtl {
    Work wk;
    SegWalk walk;
    int valid, vb, g0, g1, slot;  // the segment the CTA starts next

    // (thread 0) Step the walk to the next segment; a sequence's first segment records where
    // its partials are for the combine kernel.
    __device__ __forceinline__ void advance(int2* seg_table) {
        valid = walk.next(wk, &vb, &g0, &g1, &slot);
        if (valid && g0 == 0) {
            const int gr = wk.gran(vb);
            int np;
            if (wk.pieces)
                np = wk.npieces(vb % wk.B, wk.chunk);
            else
                np = wk.range_of(walk.seg_start + gr - 1) - (slot - vb) + 1;
            seg_table[vb] = make_int2(slot, np);
        }
    }
};
constexpr int kCtlBytes = 256;
static_assert(sizeof(SplitCtl) <= kCtlBytes, "control block");
constexpr int kBtPrefetchEntries = 1 << 14;  // block tables up to this many entries are prefetched into L2
constexpr int kFillAlone = 8;                 // ring fills of up to this many stages are issued by one thread
// A stage carries the latents of every head the CTA scans (two tensors, 8 tokens); up to this
// many elements per token (64 KB a stage) all heads are scanned together, beyond it the heads
// are split into groups scanned by different CTAs (else fewer than three stages would fit).
constexpr int kGroupLatents = 2048;
// Stages of one granule at most half of this are made two granules (16 tokens) long: a copy
// instruction costs its thread ~60-80 ns whatever its size, so small stages were bound by the
// issue of their four copies.  (Four granules per stage measured slower on the 12-layer
// backbone, 90.2 vs 85.7 us: fewer ring slots and consumer groups; eight, 197 us.)
constexpr int kSmallStageBytes = 16 << 10;

}  // namespace lrkv
