// api.cu -- the extern "C" entry points of include/lrkv.h: argument validation,
// TMA descriptor encoding, workspace carving and kernel launches on the
// caller's stream.  No allocation, no state kept between calls.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "lrkv_internal.cuh"

#include "kernels.h"
#include "mla.h"
#include "train.h"

namespace {

thread_local char g_last_error[512] = "";

lrkv_status fail(lrkv_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

lrkv_status ok() {
    g_last_error[0] = '\0';
    return LRKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxSplits = 1 << 16;

lrkv_status check_dims(const lrkv_dims* dm) {
    if (!dm) return fail(LRKV_ERR_INVALID_ARG, "dims is NULL");
    if (dm->block_size != 64) return fail(LRKV_ERR_UNSUPPORTED, "block_size %d (only 64 is supported)", dm->block_size);
    if (dm->d_h != 64 && dm->d_h != 128) return fail(LRKV_ERR_UNSUPPORTED, "d_h %d (supported: 64, 128)", dm->d_h);
    if (!(dm->r == 8 || dm->r == 16 || dm->r == 32))
        return fail(LRKV_ERR_UNSUPPORTED, "r %d (supported: 8, 16, 32)", dm->r);
    if (dm->r > dm->d_h) return fail(LRKV_ERR_UNSUPPORTED, "r %d > d_h %d", dm->r, dm->d_h);
    if (dm->H < 1 || dm->H > 128) return fail(LRKV_ERR_UNSUPPORTED, "H %d (supported: 1..128)", dm->H);
    if (dm->d < 8 || dm->d % 8 != 0) return fail(LRKV_ERR_UNSUPPORTED, "d %d (must be a positive multiple of 8)", dm->d);
    if (!(dm->softmax_scale >= 0.f) || std::isinf(dm->softmax_scale))
        return fail(LRKV_ERR_INVALID_ARG, "softmax_scale %g", (double)dm->softmax_scale);
    if (dm->d_rope != 0 && dm->d_rope != 64)
        return fail(LRKV_ERR_UNSUPPORTED, "d_rope %d (supported: 0, 64)", dm->d_rope);
    if (!(dm->rope_base >= 0.f) || std::isinf(dm->rope_base) || (dm->rope_base > 0.f && dm->rope_base <= 1.f))
        return fail(LRKV_ERR_INVALID_ARG, "rope_base %g (0 for 10000, else > 1)", (double)dm->rope_base);
    if (dm->num_splits < 0 || dm->num_splits > kMaxSplits)
        return fail(LRKV_ERR_INVALID_ARG, "num_splits %d (0 = automatic, else 1..%d)", dm->num_splits, kMaxSplits);
    return LRKV_OK;
}

// Limit of the decode split kernel's pipeline waits: about 2 s, unless the environment
// variable LRKV_DEBUG_WAIT_LIMIT_NS sets another (a debugging aid: with a short limit a wait
// that is merely slow gives up and the call reports LRKV_DEV_TIMEOUT, which lets a test see
// the expiry path run to its end on a healthy GPU).
unsigned long long decode_wait_limit_ns() {
    const char* v = std::getenv("LRKV_DEBUG_WAIT_LIMIT_NS");
    if (!v || !*v) return lrkv::kWaitLimitNs;
    char* end = nullptr;
    const unsigned long long x = std::strtoull(v, &end, 10);
    return (end && *end == '\0' && x <= lrkv::kWaitLimitNs) ? x : lrkv::kWaitLimitNs;
}

// Ranges a decode cuts the batch's cached tokens into: the caller's count, else one per SM.
int decode_ranges(const lrkv_dims* dm, int sms) { return dm->num_splits > 0 ? dm->num_splits : sms; }

// Logit scale: the caller's, else 1/sqrt of the full key width d_h + d_rope.
float logit_scale(const lrkv_dims* dm) {
    return dm->softmax_scale > 0.f ? dm->softmax_scale : 1.0f / std::sqrt((float)(dm->d_h + dm->d_rope));
}

lrkv_status check_cache(const lrkv_cache* c) {
    if (!c) return fail(LRKV_ERR_INVALID_ARG, "cache is NULL");
    if (!c->sK || !c->sV || !c->zK || !c->zV) return fail(LRKV_ERR_INVALID_ARG, "cache pool pointer is NULL");
    if (!aligned16(c->sK) || !aligned16(c->sV) || !aligned16(c->zK) || !aligned16(c->zV))
        return fail(LRKV_ERR_INVALID_ARG, "cache pool pointer not 16-byte aligned");
    if (c->num_blocks < 1 || c->num_blocks > (1 << 24))
        return fail(LRKV_ERR_INVALID_ARG, "num_blocks %d outside [1, 2^24]", c->num_blocks);
    return LRKV_OK;
}

#define LRKV_REQUIRE_PTR(p)                                                               \
    do {                                                                                  \
        if (!(p)) return fail(LRKV_ERR_INVALID_ARG, "%s is NULL", #p);                    \
        if (!aligned16(p)) return fail(LRKV_ERR_INVALID_ARG, "%s not 16-byte aligned", #p); \
    } while (0)

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};

lrkv_status device_info(DeviceInfo* di) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&di->sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&di->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return fail(LRKV_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    return LRKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix with a [box_rows][box_cols] box.
lrkv_status make_tmap(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows, CUtensorMapSwizzle swz, const char* what) {
    auto enc = encode_fn();
    if (!enc) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
    return LRKV_OK;
}

// 2-D bf16 tensor map over [rows][cols] with a row pitch of `pitch` bytes, 128-byte swizzle.
lrkv_status make_tmap_strided(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch,
                              uint32_t box_cols, uint32_t box_rows, const char* what) {
    auto enc = encode_fn();
    if (!enc) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
    return LRKV_OK;
}

// 3-D bf16 tensor map over a row-major [d2][d1][d0] array with a [1][box1][box0] box
// (box rows past d1 read as zeros).
lrkv_status make_tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                         uint32_t box1, CUtensorMapSwizzle swz, const char* what) {
    auto enc = encode_fn();
    if (!enc) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
    return LRKV_OK;
}

// 4-D bf16 tensor map over `layers` row-major [rows][cols] matrices (cols a multiple of 64),
// layer_pitch bytes apart (any valid pitch when layers == 1), that views each row as cols / 64
// parts of 64 columns, 128 bytes apart: dims {64, rows, parts, layers}.  A {64, box_rows, parts,
// 1} box then brings box_rows whole rows in one copy, laid out [part][row][64] with 128-byte
// swizzle, as cols / 64 boxes of {64, box_rows} would.
lrkv_status make_tmap_rows(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t layers,
                           uint64_t layer_pitch, uint32_t box_rows, const char* what) {
    auto enc = encode_fn();
    if (!enc) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[4] = {64, rows, cols / 64, layers};
    cuuint64_t strides[3] = {cols * 2, 128, layers > 1 ? layer_pitch : cols * 2 * rows};
    cuuint32_t box[4] = {64, box_rows, (cuuint32_t)(cols / 64), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
    return LRKV_OK;
}

// 4-D map of a latent pool [layers][rows][H][r] viewed as {128, H r / 128, rows, layers} (a token's
// latents for all heads cut into 256-byte pieces) with box {128, hl r / 128, 8, 1}: one copy brings
// the latents of hl consecutive heads (a whole number of pieces) for 8 tokens, landing as
// [token][head][r].  (Boxes one head's r values wide made 32-byte rows, which the copy engine
// moved far more slowly.)
lrkv_status make_tmap_z(CUtensorMap* m, const void* base, uint64_t H, uint64_t r, uint64_t rows, uint64_t layers,
                        uint64_t layer_pitch, uint32_t hl, const char* what) {
    auto enc = encode_fn();
    if (!enc) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    if ((H * r) % 128 != 0 || ((uint64_t)hl * r) % 128 != 0)
        return fail(LRKV_ERR_UNSUPPORTED, "%s: head group of %u x r %llu is not a whole number of 128-element pieces",
                    what, hl, (unsigned long long)r);
    cuuint64_t dims[4] = {128, H * r / 128, rows, layers};
    cuuint64_t strides[3] = {256, H * r * 2, layers > 1 ? layer_pitch : H * r * 2 * rows};
    cuuint32_t box[4] = {128, (cuuint32_t)(hl * r / 128), 8, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult res = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return fail(LRKV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)res);
    return LRKV_OK;
}

// A per-layer stride (elements) of a layer-batched call: at least the layer's own extent (layers
// do not overlap) and a multiple of 8 elements (16 bytes).  Unused when num_layers == 1.
lrkv_status check_stride(int64_t stride, uint64_t extent, int32_t num_layers, const char* what) {
    if (num_layers <= 1) return LRKV_OK;
    if (stride < 0 || (uint64_t)stride < extent || (stride & 7) != 0)
        return fail(LRKV_ERR_INVALID_ARG,
                    "layer stride of %s is %lld elements (must be a multiple of 8 and >= the layer's %llu)", what,
                    (long long)stride, (unsigned long long)extent);
    return LRKV_OK;
}

lrkv_status check_mla_dims(const lrkv_mla_dims* dm) {
    if (!dm) return fail(LRKV_ERR_INVALID_ARG, "dims is NULL");
    if (dm->block_size != 64) return fail(LRKV_ERR_UNSUPPORTED, "block_size %d (only 64 is supported)", dm->block_size);
    if (dm->d_c != 512) return fail(LRKV_ERR_UNSUPPORTED, "d_c %d (supported: 512)", dm->d_c);
    if (dm->d_rope != 64) return fail(LRKV_ERR_UNSUPPORTED, "d_rope %d (supported: 64)", dm->d_rope);
    if (dm->H < 1 || dm->H > 128) return fail(LRKV_ERR_UNSUPPORTED, "H %d (supported: 1..128)", dm->H);
    if (dm->d_head < 1 || dm->d_head > 4096) return fail(LRKV_ERR_INVALID_ARG, "d_head %d", dm->d_head);
    if (dm->d < 8 || dm->d % 8 != 0) return fail(LRKV_ERR_UNSUPPORTED, "d %d (must be a positive multiple of 8)", dm->d);
    if (!(dm->softmax_scale >= 0.f) || std::isinf(dm->softmax_scale))
        return fail(LRKV_ERR_INVALID_ARG, "softmax_scale %g", (double)dm->softmax_scale);
    if (!(dm->rope_base >= 0.f) || std::isinf(dm->rope_base) || (dm->rope_base > 0.f && dm->rope_base <= 1.f))
        return fail(LRKV_ERR_INVALID_ARG, "rope_base %g (0 for 10000, else > 1)", (double)dm->rope_base);
    return LRKV_OK;
}

int mla_pairs(const DeviceInfo& di) { return di.sms / 2 > 0 ? di.sms / 2 : 1; }

lrkv_status cuda_status(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return fail(LRKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

}  // namespace

namespace lrkv {
// Lets entry points defined in other translation units report through lrkv_last_error().
lrkv_status report_error(lrkv_status s, const char* msg) { return fail(s, "%s", msg); }
}  // namespace lrkv

extern "C" {

int lrkv_abi_version(void) { return LRKV_ABI_VERSION; }

const char* lrkv_status_string(lrkv_status s) {
    switch (s) {
        case LRKV_OK: return "ok";
        case LRKV_ERR_INVALID_ARG: return "invalid argument";
        case LRKV_ERR_UNSUPPORTED: return "unsupported shape";
        case LRKV_ERR_WORKSPACE: return "workspace too small";
        case LRKV_ERR_CUDA: return "CUDA error";
        case LRKV_ERR_DEVICE_BOUNDS: return "device-side index out of range";
        case LRKV_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char* lrkv_last_error(void) { return g_last_error; }

size_t lrkv_cache_block_bytes(const lrkv_dims* dims) {
    if (check_dims(dims) != LRKV_OK) return 0;
    return (size_t)dims->block_size * 2 * (2 * (size_t)(dims->d_h + dims->H * dims->r) + (size_t)dims->d_rope);
}

// Shared body of lrkv_append (one layer) and lrkv_append_layers.
static lrkv_status append_impl(const lrkv_dims* dims, int32_t num_layers, const lrkv_layer_strides* ls,
                               const void* X, const void* W_catT, int32_t n_tok, const int32_t* slot_mapping,
                               const int32_t* positions, const lrkv_cache* cache, uint32_t* status_dev,
                               void* stream) {
    lrkv_status s = check_dims(dims);
    if (s != LRKV_OK) return s;
    if ((s = check_cache(cache)) != LRKV_OK) return s;
    if (n_tok < 0) return fail(LRKV_ERR_INVALID_ARG, "n_tok %d < 0", n_tok);
    if (num_layers < 1) return fail(LRKV_ERR_INVALID_ARG, "num_layers %d < 1", num_layers);
    if (num_layers > 1 && !ls) return fail(LRKV_ERR_INVALID_ARG, "layer strides are NULL");
    if (n_tok == 0) return ok();
    LRKV_REQUIRE_PTR(X);
    LRKV_REQUIRE_PTR(W_catT);
    if (!slot_mapping) return fail(LRKV_ERR_INVALID_ARG, "slot_mapping is NULL");
    if (dims->d_rope > 0 && !positions)
        return fail(LRKV_ERR_INVALID_ARG, "positions is NULL but d_rope is %d", dims->d_rope);
    lrkv::AppendArgs a{};
    a.X = static_cast<const uint16_t*>(X);
    a.W = static_cast<const uint16_t*>(W_catT);
    a.slots = slot_mapping;
    a.sK = static_cast<uint16_t*>(cache->sK);
    a.sV = static_cast<uint16_t*>(cache->sV);
    a.zK = static_cast<uint16_t*>(cache->zK);
    a.zV = static_cast<uint16_t*>(cache->zV);
    a.status = status_dev;
    a.n = n_tok;
    a.d = dims->d;
    a.N = 2 * (dims->d_h + dims->H * dims->r) + dims->d_rope;
    a.d_h = dims->d_h;
    a.d_rope = dims->d_rope;
    a.rope_base = dims->rope_base > 0.f ? dims->rope_base : 10000.f;
    a.positions = dims->d_rope > 0 ? positions : nullptr;
    a.HR = dims->H * dims->r;
    a.nslots = (long long)cache->num_blocks * dims->block_size;
    a.layers = num_layers;
    if (num_layers > 1) {
        const uint64_t rows = (uint64_t)a.nslots;
        if ((s = check_stride(ls->X, (uint64_t)n_tok * a.d, num_layers, "X")) != LRKV_OK ||
            (s = check_stride(ls->W_catT, (uint64_t)a.N * a.d, num_layers, "W_catT")) != LRKV_OK ||
            (s = check_stride(ls->sK, rows * (a.d_h + a.d_rope), num_layers, "sK")) != LRKV_OK ||
            (s = check_stride(ls->sV, rows * a.d_h, num_layers, "sV")) != LRKV_OK ||
            (s = check_stride(ls->zK, rows * a.HR, num_layers, "zK")) != LRKV_OK ||
            (s = check_stride(ls->zV, rows * a.HR, num_layers, "zV")) != LRKV_OK)
            return s;
        a.ls_X = ls->X;
        a.ls_W = ls->W_catT;
        a.ls_sK = ls->sK;
        a.ls_sV = ls->sV;
        a.ls_zK = ls->zK;
        a.ls_zV = ls->zV;
    }
    if (n_tok >= lrkv::kAppendTcMinRows) {
        // the tensor-core GEMM: one launch per layer (its tensor maps are per layer)
        lrkv::AppendArgs al = a;
        al.layers = 1;
        for (int l = 0; l < num_layers; ++l) {
            al.X = a.X + l * a.ls_X;
            al.W = a.W + l * a.ls_W;
            al.sK = a.sK + l * a.ls_sK;
            al.sV = a.sV + l * a.ls_sV;
            al.zK = a.zK + l * a.ls_zK;
            al.zV = a.zV + l * a.ls_zV;
            CUtensorMap tX, tW;
            const int bn = lrkv::append_tc_block_n(a.N);
            if ((s = make_tmap(&tX, al.X, dims->d, n_tok, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "X")) != LRKV_OK)
                return s;
            if ((s = make_tmap(&tW, al.W, dims->d, a.N, 64, bn, CU_TENSOR_MAP_SWIZZLE_128B, "W_catT")) != LRKV_OK)
                return s;
            if ((s = cuda_status(lrkv::launch_append_tc(tX, tW, al, static_cast<cudaStream_t>(stream)),
                                 "lrkv_append launch")) != LRKV_OK)
                return s;
        }
        return ok();
    }
    return cuda_status(lrkv::launch_append(a, static_cast<cudaStream_t>(stream)), "lrkv_append launch");
}

lrkv_status lrkv_append(const lrkv_dims* dims, const void* X, const void* W_catT, int32_t n_tok,
                        const int32_t* slot_mapping, const int32_t* positions, const lrkv_cache* cache,
                        uint32_t* status_dev, void* stream) {
    return append_impl(dims, 1, nullptr, X, W_catT, n_tok, slot_mapping, positions, cache, status_dev, stream);
}

lrkv_status lrkv_append_layers(const lrkv_dims* dims, int32_t num_layers, const lrkv_layer_strides* strides,
                               const void* X, const void* W_catT, int32_t n_tok, const int32_t* slot_mapping,
                               const int32_t* positions, const lrkv_cache* cache, uint32_t* status_dev,
                               void* stream) {
    return append_impl(dims, num_layers, strides, X, W_catT, n_tok, slot_mapping, positions, cache, status_dev,
                       stream);
}

size_t lrkv_decode_workspace_bytes(const lrkv_dims* dims, int32_t batch) {
    if (check_dims(dims) != LRKV_OK || batch < 0) return 0;
    DeviceInfo di;
    if (device_info(&di) != LRKV_OK) return 0;
    return lrkv::decode_workspace_bytes(dims->H, dims->d_h, dims->r, batch, decode_ranges(dims, di.sms));
}

// Shared body of lrkv_decode (q~ = q B^K computed here, output B^V-projected), lrkv_decode_fused
// (q~ given by the caller, output [o_s | o_z] / l), lrkv_decode_layers (several layers) and
// lrkv_decode_partials (partials instead of an output: q~ computed, no B^V).
static lrkv_status decode_impl(const lrkv_dims* dims, int32_t num_layers, const lrkv_layer_strides* ls,
                               const void* q, const void* q_tilde, const void* BK, const void* BV,
                               const lrkv_cache* cache, const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* seq_lens, int32_t batch, void* out, void* workspace,
                               size_t workspace_bytes, uint32_t* status_dev, void* stream,
                               float* partials = nullptr) {
    const bool fused = q_tilde != nullptr;
    const char* what = partials ? "lrkv_decode_partials launch"
                                : fused ? "lrkv_decode_fused launch" : "lrkv_decode launch";
    lrkv_status s = check_dims(dims);
    if (s != LRKV_OK) return s;
    if ((s = check_cache(cache)) != LRKV_OK) return s;
    if (batch < 0) return fail(LRKV_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (num_layers < 1) return fail(LRKV_ERR_INVALID_ARG, "num_layers %d < 1", num_layers);
    if (num_layers > 1 && !ls) return fail(LRKV_ERR_INVALID_ARG, "layer strides are NULL");
    if ((long long)num_layers * batch > 65535)  // one grid row per (layer, sequence)
        return fail(LRKV_ERR_INVALID_ARG, "num_layers x batch = %lld (at most 65535)",
                    (long long)num_layers * batch);
    if (batch == 0) return ok();
    if (max_blocks_per_seq < 1 || (long long)max_blocks_per_seq * dims->block_size > (1LL << 30))
        return fail(LRKV_ERR_INVALID_ARG, "max_blocks_per_seq %d", max_blocks_per_seq);
    // the split kernel counts the call's 8-token granules in 32 bits
    if ((long long)num_layers * batch * max_blocks_per_seq * dims->block_size >= (1LL << 34))
        return fail(LRKV_ERR_INVALID_ARG, "num_layers x batch x max_blocks_per_seq x block_size = %lld (below 2^34)",
                    (long long)num_layers * batch * max_blocks_per_seq * dims->block_size);
    LRKV_REQUIRE_PTR(q);
    if (fused) {
        LRKV_REQUIRE_PTR(q_tilde);
    } else if (partials) {
        LRKV_REQUIRE_PTR(BK);
        LRKV_REQUIRE_PTR(partials);
    } else {
        LRKV_REQUIRE_PTR(BK);
        LRKV_REQUIRE_PTR(BV);
    }
    if (!partials) LRKV_REQUIRE_PTR(out);
    if (!block_table || !seq_lens) return fail(LRKV_ERR_INVALID_ARG, "block_table or seq_lens is NULL");
    const uint64_t rows = (uint64_t)cache->num_blocks * dims->block_size;
    const uint64_t dk = (uint64_t)dims->d_h + dims->d_rope;  // key row [s^K | k^R]
    const uint64_t HR = (uint64_t)dims->H * dims->r;
    lrkv::DecodeArgs a{};
    a.layers = num_layers;
    if (num_layers > 1) {
        if ((s = check_stride(ls->q, (uint64_t)batch * dims->H * dk, num_layers, "q")) != LRKV_OK ||
            (s = check_stride(ls->out, (uint64_t)batch * dims->H * dims->d_h, num_layers, "out")) != LRKV_OK ||
            (s = check_stride(ls->BK, HR * dims->d_h, num_layers, "BK")) != LRKV_OK ||
            (s = check_stride(ls->BV, HR * dims->d_h, num_layers, "BV")) != LRKV_OK ||
            (s = check_stride(ls->sK, rows * dk, num_layers, "sK")) != LRKV_OK ||
            (s = check_stride(ls->sV, rows * dims->d_h, num_layers, "sV")) != LRKV_OK ||
            (s = check_stride(ls->zK, rows * HR, num_layers, "zK")) != LRKV_OK ||
            (s = check_stride(ls->zV, rows * HR, num_layers, "zV")) != LRKV_OK)
            return s;
        a.ls_q = ls->q;
        a.ls_out = ls->out;
        a.ls_BK = ls->BK;
        a.ls_BV = ls->BV;
        a.ls_zK = ls->zK;
        a.ls_zV = ls->zV;
    }
    DeviceInfo di;
    if ((s = device_info(&di)) != LRKV_OK) return s;
    const int nvb = num_layers * batch;
    const int nranges = decode_ranges(dims, di.sms);
    const size_t need = lrkv::decode_workspace_bytes(dims->H, dims->d_h, dims->r, nvb, nranges);
    if (!workspace || ((uintptr_t)workspace & 255u))
        return fail(LRKV_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (workspace_bytes < need)
        return fail(LRKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);

    CUtensorMap tK, tV;
    const uint32_t box_rows = 8u * lrkv::decode_stage_granules(dims->H, dims->d_h, dims->r, dims->d_rope);
    if ((s = make_tmap_rows(&tK, cache->sK, dk, rows, num_layers, num_layers > 1 ? (uint64_t)ls->sK * 2 : 0,
                            box_rows, "sK")) != LRKV_OK)
        return s;
    if ((s = make_tmap_rows(&tV, cache->sV, dims->d_h, rows, num_layers, num_layers > 1 ? (uint64_t)ls->sV * 2 : 0,
                            box_rows, "sV")) != LRKV_OK)
        return s;
    if (!lrkv::decode_fits(dims->H, dims->d_h, dims->r, dims->d_rope, di.smem_optin))
        return fail(LRKV_ERR_UNSUPPORTED, "H %d x r %d: the decode's shared-memory stages do not fit on this device",
                    dims->H, dims->r);
    // Several head groups: each CTA copies its group's latent slice with a tensor map.
    const int nhg = lrkv::decode_head_groups(dims->H, dims->r);
    CUtensorMap tZK{}, tZV{};
    if (nhg > 1) {
        const uint32_t hl = (uint32_t)(dims->H / nhg);
        if ((s = make_tmap_z(&tZK, cache->zK, dims->H, dims->r, rows, num_layers,
                             num_layers > 1 ? (uint64_t)ls->zK * 2 : 0, hl, "zK")) != LRKV_OK ||
            (s = make_tmap_z(&tZV, cache->zV, dims->H, dims->r, rows, num_layers,
                             num_layers > 1 ? (uint64_t)ls->zV * 2 : 0, hl, "zV")) != LRKV_OK)
            return s;
    }

    a.q = static_cast<const uint16_t*>(q);
    a.BK = static_cast<const uint16_t*>(BK);
    a.BV = static_cast<const uint16_t*>(BV);
    a.qt_in = static_cast<const uint16_t*>(q_tilde);
    a.fused_out = fused ? 1 : 0;
    a.part_out = partials;
    a.zK = static_cast<const uint16_t*>(cache->zK);
    a.zV = static_cast<const uint16_t*>(cache->zV);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.status = status_dev;
    a.out = static_cast<uint16_t*>(out);
    a.B = batch;
    a.H = dims->H;
    a.max_pages = max_blocks_per_seq;
    a.num_blocks = cache->num_blocks;
    a.nranges = nranges;
    a.wait_ns = decode_wait_limit_ns();
    a.scale_log2 = logit_scale(dims) * 1.4426950408889634f;
    lrkv::decode_carve_workspace(&a, workspace, dims->H, dims->d_h, dims->r, nvb, nranges);
    a.nhg = nhg;
    return cuda_status(lrkv::launch_decode(tK, tV, tZK, tZV, a, dims->d_h, dims->r, dims->d_rope, di.sms,
                                           di.smem_optin,
                                           static_cast<cudaStream_t>(stream)),
                       what);
}

lrkv_status lrkv_decode(const lrkv_dims* dims, const void* q, const void* BK, const void* BV, const lrkv_cache* cache,
                        const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                        int32_t batch, void* out, void* workspace, size_t workspace_bytes, uint32_t* status_dev,
                        void* stream) {
    return decode_impl(dims, 1, nullptr, q, nullptr, BK, BV, cache, block_table, max_blocks_per_seq, seq_lens, batch,
                       out, workspace, workspace_bytes, status_dev, stream);
}

lrkv_status lrkv_decode_layers(const lrkv_dims* dims, int32_t num_layers, const lrkv_layer_strides* strides,
                               const void* q, const void* BK, const void* BV, const lrkv_cache* cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t batch, void* out, void* workspace, size_t workspace_bytes,
                               uint32_t* status_dev, void* stream) {
    return decode_impl(dims, num_layers, strides, q, nullptr, BK, BV, cache, block_table, max_blocks_per_seq,
                       seq_lens, batch, out, workspace, workspace_bytes, status_dev, stream);
}

lrkv_status lrkv_decode_fused(const lrkv_dims* dims, const void* q, const void* q_tilde, const lrkv_cache* cache,
                              const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t batch, void* out, void* workspace, size_t workspace_bytes,
                              uint32_t* status_dev, void* stream) {
    if (!q_tilde) return fail(LRKV_ERR_INVALID_ARG, "q_tilde is NULL");
    return decode_impl(dims, 1, nullptr, q, q_tilde, nullptr, nullptr, cache, block_table, max_blocks_per_seq,
                       seq_lens, batch, out, workspace, workspace_bytes, status_dev, stream);
}

lrkv_status lrkv_decode_partials(const lrkv_dims* dims, const void* q, const void* BK, const lrkv_cache* cache,
                                 const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t batch, float* partials, void* workspace, size_t workspace_bytes,
                                 uint32_t* status_dev, void* stream) {
    if (!partials) return fail(LRKV_ERR_INVALID_ARG, "partials is NULL");
    return decode_impl(dims, 1, nullptr, q, nullptr, BK, nullptr, cache, block_table, max_blocks_per_seq, seq_lens,
                       batch, nullptr, workspace, workspace_bytes, status_dev, stream, partials);
}

lrkv_status lrkv_decode_merge(const lrkv_dims* dims, int32_t num_parts, const float* partials, const void* BV,
                              int32_t batch, void* out, uint32_t* status_dev, void* stream) {
    lrkv_status s = check_dims(dims);
    if (s != LRKV_OK) return s;
    if (num_parts < 1) return fail(LRKV_ERR_INVALID_ARG, "num_parts %d < 1", num_parts);
    if (batch < 0) return fail(LRKV_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (batch == 0) return ok();
    if (batch > 65535) return fail(LRKV_ERR_INVALID_ARG, "batch %d (at most 65535)", batch);
    LRKV_REQUIRE_PTR(partials);
    LRKV_REQUIRE_PTR(BV);
    LRKV_REQUIRE_PTR(out);
    return cuda_status(lrkv::launch_decode_merge(partials, num_parts, static_cast<const uint16_t*>(BV), batch, dims->H,
                                                 dims->d_h, dims->r, static_cast<uint16_t*>(out), status_dev,
                                                 static_cast<cudaStream_t>(stream)),
                       "lrkv_decode_merge launch");
}

size_t lrkv_prefill_workspace_bytes(const lrkv_dims* dims, int32_t batch, int32_t Tq) {
    (void)batch;
    (void)Tq;
    if (check_dims(dims) != LRKV_OK) return 0;
    return 0;
}

// Shared body of lrkv_prefill (q~ = q B^K computed here, output B^V-projected) and
// lrkv_prefill_fused (q~ given by the caller, output [o_s | o_z] / l).
static lrkv_status prefill_impl(bool fused, const lrkv_dims* dims, const void* q, const void* q_tilde,
                                const void* BK, const void* BV, const lrkv_cache* cache, const int32_t* block_table,
                                int32_t max_blocks_per_seq, const int32_t* q_start, int32_t batch, int32_t Tq,
                                void* out, uint32_t* status_dev, void* stream) {
    const char* what = fused ? "lrkv_prefill_fused launch" : "lrkv_prefill launch";
    lrkv_status s = check_dims(dims);
    if (s != LRKV_OK) return s;
    if ((s = check_cache(cache)) != LRKV_OK) return s;
    if (batch < 0 || Tq < 0) return fail(LRKV_ERR_INVALID_ARG, "batch %d / Tq %d < 0", batch, Tq);
    if (batch == 0 || Tq == 0) return ok();
    if (max_blocks_per_seq < 1 || (long long)max_blocks_per_seq * dims->block_size > (1LL << 30))
        return fail(LRKV_ERR_INVALID_ARG, "max_blocks_per_seq %d", max_blocks_per_seq);
    LRKV_REQUIRE_PTR(q);
    if (fused) {
        LRKV_REQUIRE_PTR(q_tilde);
    } else {
        LRKV_REQUIRE_PTR(BK);
        LRKV_REQUIRE_PTR(BV);
    }
    LRKV_REQUIRE_PTR(out);
    if (!block_table || !q_start) return fail(LRKV_ERR_INVALID_ARG, "block_table or q_start is NULL");
    lrkv::PrefillArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.qt = static_cast<const uint16_t*>(q_tilde);
    a.BK = static_cast<const uint16_t*>(BK);
    a.BV = static_cast<const uint16_t*>(BV);
    a.sK = static_cast<const uint16_t*>(cache->sK);
    a.sV = static_cast<const uint16_t*>(cache->sV);
    a.zK = static_cast<const uint16_t*>(cache->zK);
    a.zV = static_cast<const uint16_t*>(cache->zV);
    a.block_table = block_table;
    a.q_start = q_start;
    a.status = status_dev;
    a.out = static_cast<uint16_t*>(out);
    a.B = batch;
    a.Tq = Tq;
    a.H = dims->H;
    a.max_pages = max_blocks_per_seq;
    a.num_blocks = cache->num_blocks;
    a.scale_log2 = logit_scale(dims) * 1.4426950408889634f;
    const bool tc = (dims->d_h == 64 || dims->d_h == 128) && dims->r == 16 &&
                    (dims->d_rope == 0 || (dims->d_rope == 64 && dims->d_h == 128 && !fused));
    if (tc) {
        lrkv::PrefillMaps mp;
        const uint64_t dh = (uint64_t)dims->d_h, dk = dh + (uint64_t)dims->d_rope;
        const uint64_t rows = (uint64_t)cache->num_blocks * dims->block_size;
        const uint64_t HR = (uint64_t)dims->H * dims->r;
        if ((s = make_tmap(&mp.q, q, (uint64_t)dims->H * dk, (uint64_t)batch * Tq, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B, "q")) != LRKV_OK ||
            (s = make_tmap(&mp.sK, cache->sK, dk, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "sK")) != LRKV_OK ||
            (s = make_tmap(&mp.sV, cache->sV, dh, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "sV")) != LRKV_OK ||
            (s = make_tmap(&mp.zK, cache->zK, HR, rows, 16, 64, CU_TENSOR_MAP_SWIZZLE_32B, "zK")) != LRKV_OK ||
            (s = make_tmap(&mp.zV, cache->zV, HR, rows, 16, 64, CU_TENSOR_MAP_SWIZZLE_32B, "zV")) != LRKV_OK)
            return s;
        if (fused) {
            s = make_tmap(&mp.qt, q_tilde, HR, (uint64_t)batch * Tq, 16, 128, CU_TENSOR_MAP_SWIZZLE_32B, "q_tilde");
            mp.BK = mp.qt;
        } else {
            s = make_tmap(&mp.BK, BK, 16, (uint64_t)dims->H * dh, 16, (uint32_t)dh, CU_TENSOR_MAP_SWIZZLE_32B, "BK");
            mp.qt = mp.BK;
        }
        if (s != LRKV_OK) return s;
        return cuda_status(lrkv::launch_prefill_tc(mp, a, dims->d_h, dims->d_rope, static_cast<cudaStream_t>(stream)),
                           what);
    }
    return cuda_status(lrkv::launch_prefill(a, dims->d_h, dims->r, dims->d_rope, static_cast<cudaStream_t>(stream)),
                       what);
}

lrkv_status lrkv_prefill(const lrkv_dims* dims, const void* q, const void* BK, const void* BV, const lrkv_cache* cache,
                         const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* q_start, int32_t batch,
                         int32_t Tq, void* out, void* workspace, size_t workspace_bytes, uint32_t* status_dev,
                         void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    return prefill_impl(false, dims, q, nullptr, BK, BV, cache, block_table, max_blocks_per_seq, q_start, batch, Tq, out,
                        status_dev, stream);
}

lrkv_status lrkv_prefill_fused(const lrkv_dims* dims, const void* q, const void* q_tilde, const lrkv_cache* cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* q_start,
                               int32_t batch, int32_t Tq, void* out, uint32_t* status_dev, void* stream) {
    return prefill_impl(true, dims, q, q_tilde, nullptr, nullptr, cache, block_table, max_blocks_per_seq, q_start, batch,
                        Tq, out, status_dev, stream);
}

// ------------------------------------------------------------------ training-time projections
static lrkv_status check_train(const lrkv_dims* dims, int32_t n_tok) {
    lrkv_status s = check_dims(dims);
    if (s != LRKV_OK) return s;
    if (dims->d_rope != 0) return fail(LRKV_ERR_UNSUPPORTED, "training projections with d_rope %d", dims->d_rope);
    if (n_tok < 0) return fail(LRKV_ERR_INVALID_ARG, "n_tok %d < 0", n_tok);
    return LRKV_OK;
}

// Split-K factor of dB_h = dK_h^T R_h (a 128 x 128 tile per head over all tokens).
static int train_dB_split(int H, int n_tok, int sms) {
    int ks = (2 * sms + H - 1) / H;
    const int maxk = (n_tok + 255) / 256;
    ks = ks > maxk ? maxk : ks;
    ks = ks > 8 ? 8 : ks;
    return ks < 1 ? 1 : ks;
}

size_t lrkv_train_workspace_bytes(const lrkv_dims* dims, int32_t n_tok) {
    if (check_train(dims, n_tok) != LRKV_OK) return 0;
    DeviceInfo di;
    if (device_info(&di) != LRKV_OK) return 0;
    const size_t Ncat = (size_t)dims->d_h + (size_t)dims->H * dims->r;
    const size_t gc = ((size_t)n_tok * Ncat * 2 + 255) & ~(size_t)255;
    const size_t bt = ((size_t)dims->H * dims->r * dims->d_h * 2 + 255) & ~(size_t)255;
    const size_t split = (size_t)train_dB_split(dims->H, n_tok, di.sms) * 128 * 64;
    const size_t tiles = (size_t)((n_tok + 127) / 128) * 128 * 16;  // partials of the folded dB
    return gc + bt + 256 + (size_t)dims->H * (split > tiles ? split : tiles) * 4;
}

// Output map of a tcgen05 GEMM: set g->tma_out when the output can go through TMA (16-byte
// aligned base and strides), else the epilogue stores directly.
static void train_out_map(lrkv::GemmArgs* g, CUtensorMap* tC) {
    g->tma_out = 0;
    const uint64_t zs = g->nbatch > 1 ? (uint64_t)g->c_zstride * 2 : (uint64_t)g->ldc * 2;
    if (((uintptr_t)g->C & 15u) || ((uint64_t)g->ldc * 2) % 16 || zs % 16 || zs == 0) return;
    auto enc = encode_fn();
    if (!enc) return;
    cuuint64_t dims[3] = {(cuuint64_t)g->N, (cuuint64_t)g->nbatch, (cuuint64_t)g->M};
    cuuint64_t strides[2] = {zs, (cuuint64_t)g->ldc * 2};
    cuuint32_t box[3] = {32, 1, 32};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(tC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, g->C, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return;
    g->tma_out = 1;
}

// C = A . B on the tensor cores (see train.h); bf16 outputs go through TMA when they can.
static cudaError_t train_gemm(const CUtensorMap& tA, const CUtensorMap& tB, lrkv::GemmArgs g, int bn, bool a_mn,
                              bool b_mn, bool out_f32, cudaStream_t st, const CUtensorMap* tB2 = nullptr) {
    CUtensorMap tC = tA;
    g.a_mn = a_mn;
    g.b_mn = b_mn;
    if (!out_f32) train_out_map(&g, &tC);
    return lrkv::launch_tgemm(tA, tB, tB2 ? *tB2 : tB, tC, g, bn, out_f32, st);
}

lrkv_status lrkv_train_forward(const lrkv_dims* dims, const void* X, const void* W_T, const void* B, int32_t n_tok,
                               void* Y, void* K, uint32_t* status_dev, void* stream) {
    lrkv_status s = check_train(dims, n_tok);
    if (s != LRKV_OK) return s;
    if (n_tok == 0) return ok();
    LRKV_REQUIRE_PTR(X);
    LRKV_REQUIRE_PTR(W_T);
    LRKV_REQUIRE_PTR(B);
    LRKV_REQUIRE_PTR(Y);
    LRKV_REQUIRE_PTR(K);
    const int H = dims->H, d_h = dims->d_h, r = dims->r, d = dims->d, Ncat = d_h + H * r;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap tX, tW, tY, tB;
    if ((s = make_tmap(&tX, X, d, n_tok, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "X")) != LRKV_OK ||
        (s = make_tmap(&tW, W_T, d, Ncat, 64, 160, CU_TENSOR_MAP_SWIZZLE_128B, "W_T")) != LRKV_OK ||
        (s = make_tmap(&tY, Y, Ncat, n_tok, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "Y")) != LRKV_OK ||
        (s = make_tmap(&tB, B, r, (uint64_t)H * d_h, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "B")) != LRKV_OK)
        return s;
    // Y = [S | R_1 .. R_H] = X W_T^T
    lrkv::GemmArgs g{};
    g.C = Y; g.ldc = Ncat; g.M = n_tok; g.N = Ncat; g.K = d; g.nbatch = 1; g.ksplit = 1; g.status = status_dev;
    cudaError_t e = train_gemm(tX, tW, g, 160, false, false, false, st);
    if (e != cudaSuccess) return cuda_status(e, "lrkv_train_forward launch");
    // K_h = [S | R_h] [I ; B_h^T], one batch per head: the first d_h K columns are S (Y columns
    // [0, d_h)) against the identity, the rest R_h (Y columns d_h + h r ..) against B_h as [d_h][r]
    const void* ident = lrkv::train_identity();
    if (!ident) return fail(LRKV_ERR_CUDA, "identity table unavailable");
    CUtensorMap tI;
    if ((s = make_tmap_strided(&tI, ident, d_h, d_h, 256, 64, 128, "identity")) != LRKV_OK) return s;
    lrkv::GemmArgs x{};
    x.C = K; x.ldc = H * d_h; x.c_zstride = d_h; x.M = n_tok; x.N = d_h; x.K = d_h + r; x.kfix = d_h;
    x.a_x0 = d_h; x.a_zx = r; x.b_zy = d_h; x.nbatch = H; x.ksplit = 1; x.status = status_dev;
    return cuda_status(train_gemm(tY, tB, x, 128, false, false, false, st, &tI), "lrkv_train_forward launch");
}

lrkv_status lrkv_train_backward(const lrkv_dims* dims, const void* X, const void* W_T, const void* B, const void* Y,
                                const void* dK, int32_t n_tok, void* dX, void* dW_T, void* dB, void* workspace,
                                size_t workspace_bytes, uint32_t* status_dev, void* stream) {
    lrkv_status s = check_train(dims, n_tok);
    if (s != LRKV_OK) return s;
    if (n_tok == 0) return ok();
    LRKV_REQUIRE_PTR(X);
    LRKV_REQUIRE_PTR(W_T);
    LRKV_REQUIRE_PTR(B);
    LRKV_REQUIRE_PTR(Y);
    LRKV_REQUIRE_PTR(dK);
    LRKV_REQUIRE_PTR(dX);
    LRKV_REQUIRE_PTR(dW_T);
    LRKV_REQUIRE_PTR(dB);
    DeviceInfo di;
    if ((s = device_info(&di)) != LRKV_OK) return s;
    const int H = dims->H, d_h = dims->d_h, r = dims->r, d = dims->d, Ncat = d_h + H * r;
    const int ks = train_dB_split(H, n_tok, di.sms);
    const size_t gc_bytes = ((size_t)n_tok * Ncat * 2 + 255) & ~(size_t)255;
    const size_t bt_bytes = ((size_t)H * r * d_h * 2 + 255) & ~(size_t)255;
    const int ntiles = (n_tok + 127) / 128;
    const bool fold_dB = lrkv::dk_pass_folds_dB(H, d_h, r);
    const size_t pfl = fold_dB ? (size_t)ntiles * 128 * 16 : (size_t)ks * 128 * 64;  // floats per head
    const size_t need = gc_bytes + bt_bytes + 256 + (size_t)H * pfl * 4;
    if (!workspace || ((uintptr_t)workspace & 255u))
        return fail(LRKV_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (workspace_bytes < need) return fail(LRKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    uint16_t* Gc = static_cast<uint16_t*>(workspace);
    uint16_t* BT = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + gc_bytes);
    int* ctr = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + gc_bytes + bt_bytes);
    float* P = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + gc_bytes + bt_bytes + 256);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap tdK_k, tdK_mn, tB_mn, tY_mn, tGc_mn, tGc_k, tX_mn, tW_mn;
    const uint64_t HD = (uint64_t)H * d_h;
    if ((s = make_tmap(&tdK_k, dK, HD, n_tok, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "dK")) != LRKV_OK ||
        (s = make_tmap(&tdK_mn, dK, HD, n_tok, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "dK")) != LRKV_OK ||
        (s = make_tmap(&tB_mn, B, r, HD, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "B")) != LRKV_OK ||
        (s = make_tmap(&tY_mn, Y, Ncat, n_tok, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "Y")) != LRKV_OK ||
        (s = make_tmap(&tGc_mn, Gc, Ncat, n_tok, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "Gc")) != LRKV_OK ||
        (s = make_tmap(&tGc_k, Gc, Ncat, n_tok, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "Gc")) != LRKV_OK ||
        (s = make_tmap(&tX_mn, X, d, n_tok, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "X")) != LRKV_OK ||
        (s = make_tmap(&tW_mn, W_T, d, Ncat, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "W_T")) != LRKV_OK)
        return s;
    cudaError_t e;
    lrkv::GemmArgs g{};
    if (lrkv::dk_pass_supported(H, d_h, r)) {
        // one pass over dK: Gc[:, 0:d_h] = G = sum_h dK_h and Gc[:, d_h + h r ..] = dR_h = dK_h B_h
        CUtensorMap tBT, tR = tdK_k;
        if ((s = make_tmap(&tBT, BT, d_h, (uint64_t)H * r, 64, r, CU_TENSOR_MAP_SWIZZLE_128B, "B^T")) != LRKV_OK ||
            (fold_dB && (s = make_tmap(&tR, Y, Ncat, n_tok, 16, 128, CU_TENSOR_MAP_SWIZZLE_32B, "R")) != LRKV_OK))
            return s;
        lrkv::DkArgs da{};
        da.Gc = Gc; da.ldg = Ncat; da.n = n_tok; da.H = H; da.d_h = d_h; da.r = r; da.status = status_dev;
        // dB_h's per-tile partials too (the same dK_h tiles against R_h), summed in tile order
        da.dBp = fold_dB ? P : nullptr;
        da.rx0 = d_h;
        if ((e = lrkv::launch_dk_pass(tdK_k, tBT, tR, static_cast<const uint16_t*>(B), BT, da, st)) != cudaSuccess)
            return cuda_status(e, "lrkv_train_backward launch");
    } else {
        // Gc[:, 0:d_h] = G = sum_h dK_h
        if ((e = lrkv::launch_head_sum(static_cast<const uint16_t*>(dK), Gc, n_tok, H, d_h, Ncat, st)) != cudaSuccess)
            return cuda_status(e, "lrkv_train_backward launch");
        // Gc[:, d_h + h r ..] = dR_h = dK_h B_h  (A = dK_h K-major, B = B_h read [d_h (K)][r (N)])
        g.C = Gc + d_h; g.ldc = Ncat; g.c_zstride = r; g.M = n_tok; g.N = r; g.K = d_h;
        g.a_zx = d_h; g.b_zy = d_h; g.nbatch = H; g.ksplit = 1; g.status = status_dev;
        if ((e = train_gemm(tdK_k, tB_mn, g, 128, false, true, false, st)) != cudaSuccess)
            return cuda_status(e, "lrkv_train_backward launch");
    }
    if (fold_dB) {
        if ((e = lrkv::launch_dB_reduce(P, static_cast<uint16_t*>(dB), H, ntiles, d_h, r, 16, st)) != cudaSuccess)
            return cuda_status(e, "lrkv_train_backward launch");
    } else {
        // dB_h = dK_h^T R_h: split-K partials (A = dK read [n (K)][d_h (M)], B = R_h read [n (K)][r (N)])
        g = lrkv::GemmArgs{};
        g.C = P; g.M = d_h; g.N = r; g.K = n_tok; g.a_zx = d_h; g.b_x0 = d_h; g.b_zx = r; g.nbatch = H;
        g.ksplit = ks; g.status = status_dev;
        if ((e = train_gemm(tdK_mn, tY_mn, g, 64, true, true, true, st)) != cudaSuccess ||
            (e = lrkv::launch_dB_reduce(P, static_cast<uint16_t*>(dB), H, ks, d_h, r, 64, st)) != cudaSuccess)
            return cuda_status(e, "lrkv_train_backward launch");
    }
    // One launch for both products of Gc, whose CTAs take tiles from a shared queue: the long
    // tiles of dW_T first (fewer than the SMs), the short tiles of dX filling the other SMs.
    //   dW_T = Gc^T X  ([d_h + H r][d]; A = Gc read [n (K)][Ncat (M)], B = X read [n (K)][d (N)])
    //   dX = Gc W_T    (A = Gc K-major, B = W_T read [Ncat (K)][d (N)])
    lrkv::GemmArgs gg[2] = {};
    gg[0].C = dW_T; gg[0].ldc = d; gg[0].M = Ncat; gg[0].N = d; gg[0].K = n_tok; gg[0].a_mn = 1; gg[0].b_mn = 1;
    gg[1].C = dX; gg[1].ldc = d; gg[1].M = n_tok; gg[1].N = d; gg[1].K = Ncat; gg[1].a_mn = 0; gg[1].b_mn = 1;
    CUtensorMap tA2[2] = {tGc_mn, tGc_k}, tB2m[2] = {tX_mn, tW_mn}, tC2[2];
    for (int i = 0; i < 2; ++i) {
        gg[i].nbatch = 1; gg[i].ksplit = 1; gg[i].status = status_dev;
        train_out_map(&gg[i], &tC2[i]);
    }
    if (gg[0].tma_out && gg[1].tma_out)
        return cuda_status(lrkv::launch_tgemm2(tA2, tB2m, tC2, gg, 256, ctr, st), "lrkv_train_backward launch");
    if ((e = train_gemm(tGc_mn, tX_mn, gg[0], 256, true, true, false, st)) != cudaSuccess)
        return cuda_status(e, "lrkv_train_backward launch");
    return cuda_status(train_gemm(tGc_k, tW_mn, gg[1], 256, false, true, false, st), "lrkv_train_backward launch");
}

size_t lrkv_mla_cache_block_bytes(const lrkv_mla_dims* dims) {
    if (check_mla_dims(dims) != LRKV_OK) return 0;
    return (size_t)dims->block_size * 2 * (size_t)(dims->d_c + dims->d_rope);
}

lrkv_status lrkv_mla_append(const lrkv_mla_dims* dims, const void* X, const void* W_T, int32_t n_tok,
                            const int32_t* slot_mapping, const int32_t* positions, void* kv, int32_t num_blocks,
                            uint32_t* status_dev, void* stream) {
    lrkv_status s = check_mla_dims(dims);
    if (s != LRKV_OK) return s;
    if (n_tok < 0) return fail(LRKV_ERR_INVALID_ARG, "n_tok %d < 0", n_tok);
    if (n_tok == 0) return ok();
    LRKV_REQUIRE_PTR(X);
    LRKV_REQUIRE_PTR(W_T);
    LRKV_REQUIRE_PTR(kv);
    if (num_blocks < 1 || num_blocks > (1 << 24)) return fail(LRKV_ERR_INVALID_ARG, "num_blocks %d", num_blocks);
    if (!slot_mapping || !positions) return fail(LRKV_ERR_INVALID_ARG, "slot_mapping or positions is NULL");
    // The cache row [c | k^R] is the shared key row of the append kernels with d_h = d_c and no
    // value or per-head columns: columns [0, d_c) plain, [d_c, d_c + d_rope) rotated.
    uint16_t* pool = static_cast<uint16_t*>(kv);
    lrkv::AppendArgs a{};
    a.X = static_cast<const uint16_t*>(X);
    a.W = static_cast<const uint16_t*>(W_T);
    a.slots = slot_mapping;
    a.positions = positions;
    a.sK = pool;
    a.sV = a.zK = a.zV = pool;  // never addressed: every column maps into the key row
    a.status = status_dev;
    a.n = n_tok;
    a.d = dims->d;
    a.N = dims->d_c + dims->d_rope;
    a.d_h = dims->d_c;
    a.HR = 0;
    a.d_rope = dims->d_rope;
    a.rope_base = dims->rope_base > 0.f ? dims->rope_base : 10000.f;
    a.nslots = (long long)num_blocks * dims->block_size;
    if (n_tok >= lrkv::kAppendTcMinRows) {
        CUtensorMap tX, tW;
        const int bn = lrkv::append_tc_block_n(a.N);
        if ((s = make_tmap(&tX, X, dims->d, n_tok, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "X")) != LRKV_OK) return s;
        if ((s = make_tmap(&tW, W_T, dims->d, a.N, 64, bn, CU_TENSOR_MAP_SWIZZLE_128B, "W_T")) != LRKV_OK) return s;
        return cuda_status(lrkv::launch_append_tc(tX, tW, a, static_cast<cudaStream_t>(stream)),
                           "lrkv_mla_append launch");
    }
    return cuda_status(lrkv::launch_append(a, static_cast<cudaStream_t>(stream)), "lrkv_mla_append launch");
}

size_t lrkv_mla_decode_workspace_bytes(const lrkv_mla_dims* dims, int32_t batch) {
    if (check_mla_dims(dims) != LRKV_OK || batch < 0) return 0;
    DeviceInfo di;
    if (device_info(&di) != LRKV_OK) return 0;
    return lrkv::mla_workspace_bytes(dims->H, batch, mla_pairs(di));
}

lrkv_status lrkv_mla_decode(const lrkv_mla_dims* dims, const void* q, const void* kv, int32_t num_blocks,
                            const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            int32_t batch, void* out, void* workspace, size_t workspace_bytes,
                            uint32_t* status_dev, void* stream) {
    lrkv_status s = check_mla_dims(dims);
    if (s != LRKV_OK) return s;
    if (batch < 0) return fail(LRKV_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (batch == 0) return ok();
    if (num_blocks < 1 || num_blocks > (1 << 24)) return fail(LRKV_ERR_INVALID_ARG, "num_blocks %d", num_blocks);
    if (max_blocks_per_seq < 1 || (long long)max_blocks_per_seq * dims->block_size > (1LL << 30))
        return fail(LRKV_ERR_INVALID_ARG, "max_blocks_per_seq %d", max_blocks_per_seq);
    LRKV_REQUIRE_PTR(q);
    LRKV_REQUIRE_PTR(kv);
    LRKV_REQUIRE_PTR(out);
    if (!block_table || !seq_lens) return fail(LRKV_ERR_INVALID_ARG, "block_table or seq_lens is NULL");
    DeviceInfo di;
    if ((s = device_info(&di)) != LRKV_OK) return s;
    lrkv::MlaArgs a{};
    a.npairs = mla_pairs(di);
    const size_t need = lrkv::mla_workspace_bytes(dims->H, batch, a.npairs);
    if (!workspace || ((uintptr_t)workspace & 255u))
        return fail(LRKV_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (workspace_bytes < need) return fail(LRKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    const uint64_t dk = (uint64_t)dims->d_c + dims->d_rope;
    CUtensorMap tQ, tQr, tKV, tKVr;
    const uint64_t rows = (uint64_t)num_blocks * dims->block_size;
    if ((s = make_tmap_3d(&tQ, q, dk, dims->H, batch, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "q")) != LRKV_OK ||
        (s = make_tmap_3d(&tQr, q, dk, dims->H, batch, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B, "q^R")) != LRKV_OK ||
        (s = make_tmap(&tKV, kv, dk, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "kv")) != LRKV_OK ||
        (s = make_tmap(&tKVr, kv, dk, rows, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B, "k^R")) != LRKV_OK)
        return s;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.status = status_dev;
    a.out = static_cast<uint16_t*>(out);
    a.B = batch;
    a.H = dims->H;
    a.max_pages = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.pmax = a.npairs > batch ? a.npairs : batch;
    const float scale = dims->softmax_scale > 0.f ? dims->softmax_scale
                                                  : 1.0f / std::sqrt((float)(dims->d_head + dims->d_rope));
    a.scale_log2 = scale * 1.4426950408889634f;
    lrkv::mla_carve_workspace(&a, workspace);
    return cuda_status(lrkv::launch_mla_decode(tQ, tQr, tKV, tKVr, a, static_cast<cudaStream_t>(stream)),
                       "lrkv_mla_decode launch");
}

}  // extern "C"
