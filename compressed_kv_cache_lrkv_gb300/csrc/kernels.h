// kernels.h -- argument blocks and launchers shared between the C-ABI layer
// (api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lrkv {

struct AppendArgs {
    const uint16_t* X;      // [n][d]
    const uint16_t* W;      // [N][d], rows [W_s^K | W^KR | W_s^V | U^K | U^V]
    const int32_t* slots;   // [n]
    const int32_t* positions;  // [n] token positions (for the positional key), or null without one
    uint16_t *sK, *sV, *zK, *zV;  // sK rows are d_h + d_rope wide: [s^K | k^R]
    uint32_t* status;
    int n, d, N, d_h, HR;
    int d_rope;             // width of the shared positional key (0: none)
    float rope_base;
    long long nslots;       // num_blocks * block_size
    // Several layers in one launch (blockIdx.z = layer): element strides between consecutive
    // layers' X, W and cache pools (slots and positions are shared by the layers).
    int layers;
    long long ls_X, ls_W, ls_sK, ls_sV, ls_zK, ls_zV;
};

// Decode over `layers` layers of B sequences at once: virtual sequence vb = layer * B + b
// (every layer shares the block table and the lengths); per-layer tensors are found at
// the element strides ls_* from layer 0's (sK, sV through the layer coordinate of their
// 3-D tensor maps).
struct DecodeArgs {
    const uint16_t* q;     // [B][H][D_H + D_R] per layer
    const uint16_t* BK;    // [H][D_H][R] per layer
    const uint16_t* BV;    // [H][D_H][R] per layer
    const uint16_t* zK;    // [nb*64][H][R] per layer
    const uint16_t* zV;
    const int32_t* block_table;  // [B][max_pages]
    const int32_t* seq_lens;     // [B]
    float* part_ml;   // [H][pmax][2]  running max (log2 domain) and sum
    float* part_acc;  // [H][pmax][D_H + R]
    float* qt;        // [layers * B][H][R]  q~ = q B^K, fp32
    int2* seg_table;  // [layers * B] first partial slot and slot count of each virtual sequence
    const uint16_t* qt_in;  // [B][H][R] bf16 q~ supplied by the caller (absorbed query weights), or null
    uint32_t* status;
    uint16_t* out;    // [B][H][D_H], or [B][H][D_H + R] = [o_s | o_z] / l when fused_out, per layer
    int fused_out;    // 1: no B^V up-projection (absorbed into the output projection)
    int B, H, max_pages, num_blocks;
    int layers;
    long long ls_q, ls_qt, ls_BK, ls_BV, ls_zK, ls_zV, ls_out;
    int nranges;       // pieces of work the batch's cached tokens are cut into (CTA iterations)
    int bubble;        // granules a pipeline drain-and-refill costs (chooses how the work is cut)
    int ng, nslot, stage_bytes;
    int nhg;           // head groups: each (layer, sequence) is scanned as nhg virtual sequences of H / nhg heads
    int gpst;          // 8-token granules per pipeline stage (1 or 2)
    int pmax;          // partial slots per head in the workspace (layers * B * nhg + nranges)
    float scale_log2;  // softmax scale * log2(e)
    unsigned long long wait_ns;  // limit of the split kernel's pipeline waits (a debugging aid may shorten it)
    // Partials out (a token-range split of the sequences): when set, the combine writes each
    // (sequence, head)'s merged, unnormalised [acc_s | acc_z | m | l] ([B][H][D_H + R + 2],
    // m in the log2 domain) here instead of out, and no B^V is read.
    float* part_out;
};

struct PrefillArgs {
    const uint16_t *q, *BK, *BV;        // q [B][Tq][H][D_H]; B* [H][D_H][R]
    // Absorbed weights when non-null: q~ [B][Tq][H][R] given (B^K, B^V unused) and
    // out [B][Tq][H][D_H + R] = [o_s | o_z] / l.
    const uint16_t* qt;
    const uint16_t *sK, *sV, *zK, *zV;  // cache pools
    const int32_t* block_table;         // [B][max_pages]
    const int32_t* q_start;             // [B]
    uint32_t* status;
    uint16_t* out;                      // [B][Tq][H][D_H] (absorbed: [B][Tq][H][D_H + R])
    int B, Tq, H, max_pages, num_blocks;
    float scale_log2;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
// Tensor-core path (rows >= kAppendTcMinRows): X and W_cat^T tensor maps with a
// {64, 128} and {64, append_tc_block_n(N)} box, 128-byte swizzle.
constexpr int kAppendTcMinRows = 64;
int append_tc_block_n(int N);
cudaError_t launch_append_tc(const CUtensorMap& tmX, const CUtensorMap& tmW, const AppendArgs& a,
                             cudaStream_t stream);

// Head groups of the decode scan: 1 while a stage's latents for all heads (8 tokens x H r
// elements, two tensors) fit in 64 KB; else the fewest groups (2, 4 or 8, dividing H into
// whole 128-element pieces of a token's latents) that bring a group's share within that.
int decode_head_groups(int H, int R);
// 8-token granules per stage of the decode scan (1, or 2 for small stages); the s^K, s^V maps'
// box is 8 x this many rows.
int decode_stage_granules(int H, int D_H, int R, int D_R);
// Whether the split kernel's shared-memory ring (at least two stages) fits in smem_limit bytes.
bool decode_fits(int H, int D_H, int R, int D_R, int smem_limit);
// Workspace of a decode over nvb = layers * B (layer, sequence) pairs cut into `nranges` ranges.
size_t decode_workspace_bytes(int H, int D_H, int R, int nvb, int nranges);
void decode_carve_workspace(DecodeArgs* a, void* ws, int H, int D_H, int R, int nvb, int nranges);
// tK, tV: 4-D maps {64, nb * 64, (d_h (+ d_rope)) / 64, layers}, box {64, 8 g, parts, 1} (g the stage's
// granules), 128-byte swizzle
// (the parts dimension steps 128 bytes along a row).  tZK, tZV (used with several head groups):
// 4-D maps {128, H r / 128, nb * 64, layers} of z^K, z^V, box {128, (H / groups) r / 128, 8, 1},
// no swizzle.
// The split kernel runs on min(nranges, sms) CTAs.
cudaError_t launch_decode(const CUtensorMap& tK, const CUtensorMap& tV, const CUtensorMap& tZK,
                          const CUtensorMap& tZV, DecodeArgs a, int D_H, int R, int D_R, int sms, int smem_limit,
                          cudaStream_t stream);

// The split-K scan on the tensor cores (H = 128, d_h = 128, no positional key, one head group):
// launched in place of the CUDA-core scan by launch_decode; smem_bytes from decode_tc_smem_bytes.
int decode_tc_smem_bytes(int nslot, int stage_bytes);
template <int R>
cudaError_t launch_decode_tc_split(const CUtensorMap& tK, const CUtensorMap& tV, const DecodeArgs& a, int grid,
                                   int smem_bytes, bool pdl, cudaStream_t stream);

// Log-sum-exp merge of nparts decode partials ([nparts][B][H][d_h + r + 2], as the combine
// writes them with part_out) and the B^V up-projection: out [B][H][d_h] bf16.
cudaError_t launch_decode_merge(const float* parts, int nparts, const uint16_t* BV, int B, int H, int d_h, int r,
                                uint16_t* out, uint32_t* status, cudaStream_t stream);

cudaError_t launch_prefill(const PrefillArgs& a, int D_H, int R, int D_R, cudaStream_t stream);

// Tensor-core prefill (d_h = 64 or 128 with r = 16; d_rope = 64 with d_h = 128 and no absorbed
// weights).  Maps: q as [B*Tq][H*(d_h + d_rope)] box {64,128} and s^K ([s^K | k^R]), s^V pools
// [nb*64][d_h + d_rope], [nb*64][d_h] box {64,64}, all 128-byte swizzle; z^K, z^V
// pools [nb*64][H*r] box {16,64} and B^K as [H*d_h][r] box {16,d_h}, 32-byte swizzle;
// with absorbed weights, q~ as [B*Tq][H*r] box {16,128}, 32-byte swizzle, in place of B^K.
struct PrefillMaps {
    CUtensorMap q, sK, sV, zK, zV, BK, qt;
};
cudaError_t launch_prefill_tc(const PrefillMaps& maps, const PrefillArgs& a, int d_h, int d_rope, cudaStream_t stream);

}  // namespace lrkv
