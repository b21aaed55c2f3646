// mla.h -- internal interface of the multi-head latent attention decode kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lrkv {

// Absorbed MLA decode over a paged cache of rows [c | k^R] (d_c = 512, d_rope = 64).
struct MlaArgs {
    const int32_t* block_table;  // [B][max_pages]
    const int32_t* seq_lens;     // [B]
    uint32_t* status;            // LRKV_DEV_* bits (may be null)
    uint16_t* out;               // [B][H][512] bf16
    float* part_ml;              // [H][pmax][2]   running max (log2 units) and sum per split
    float* part_acc;             // [H][pmax][512] unnormalised sum_t p_t c_t per split
    int* seq_first;              // [B] first split of each sequence (written by the split kernel)
    int* seq_count;              // [B] its number of splits (0: length out of range)
    int B, H, max_pages, num_blocks;
    int npairs;                  // CTA pairs (clusters) of the split kernel
    int pmax;                    // max(npairs, B): split slots per head
    float scale_log2;            // logit scale * log2(e)
};

size_t mla_workspace_bytes(int H, int B, int npairs);
void mla_carve_workspace(MlaArgs* a, void* ws);
// tmQ / tmKV: 64-column boxes (128-byte swizzle) of q and the cache; tmQr / tmKVr: 32-column
// boxes (64-byte swizzle) of their positional-key columns.
cudaError_t launch_mla_decode(const CUtensorMap& tmQ, const CUtensorMap& tmQr, const CUtensorMap& tmKV,
                              const CUtensorMap& tmKVr, const MlaArgs& a, cudaStream_t stream);

}  // namespace lrkv
