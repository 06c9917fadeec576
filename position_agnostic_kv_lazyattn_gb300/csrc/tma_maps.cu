// Host-side construction of the TMA tensor maps over a pool's K and V buffers.
#include <cudaTypedefs.h>
#include <limits.h>

#include "internal.h"

namespace lazyattn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode_one(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, void* base, uint64_t rows, int d) {
    cuuint64_t gdim[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kPage};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same pool as a 4-D tensor {D, slot, KV head, page} (strides 2 B, D * 2 B,
// 16 * D * 2 B, Hkv * 16 * D * 2 B) with boxes {64, 16, 1, run}: one box holds
// half the dims of `run` consecutive pages of one KV head, rows ordered
// (page, slot) exactly as `run` 2-D page boxes side by side.
bool encode_run(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, void* base, uint64_t pages, int hkv, int d,
                uint32_t run) {
    cuuint64_t gdim[4] = {(cuuint64_t)d, (cuuint64_t)kPage, (cuuint64_t)hkv, (cuuint64_t)pages};
    cuuint64_t gstride[3] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * kPage, (cuuint64_t)d * 2 * kPage * hkv};
    cuuint32_t box[4] = {64, (cuuint32_t)kPage, 1, run};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The paired position table (rows of D floats, (cos f, cos f+1, sin f, sin f+1)
// for even f, one row per position) as a 3-D fp32 tensor {D, 16, max_position / 16} (strides 4 B,
// 2 D B, 32 D B): a box {D, 1, pages} at (0, t % 16, t / 16) holds the rows of
// positions t, t + 16, ..., i.e. the start rows of `pages` pages that follow
// each other at consecutive positions. Positions past the last whole
// block of 16 are outside the view (callers copy those rows one by one).
bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, void* base, int32_t max_position, int d,
                 uint32_t pages) {
    cuuint64_t gdim[3] = {(cuuint64_t)d, (cuuint64_t)kPage, (cuuint64_t)(max_position / kPage)};
    cuuint64_t gstride[2] = {(cuuint64_t)d * 4, (cuuint64_t)d * 4 * kPage};
    cuuint32_t box[3] = {(cuuint32_t)d, 1, pages};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_pool_maps(lazyattn_pool& p) {
    p.have_maps = false;
    p.have_rmap = false;
    if (p.d.dtype != LAZYATTN_BF16) return false;
    const uint64_t rows = (uint64_t)p.d.num_pages * (uint64_t)p.d.n_kv_heads * kPage;
    if (rows + kPage > (uint64_t)INT_MAX) return false;
    auto enc = get_encoder();
    if (!enc) return false;
    if (!encode_one(enc, &p.kmap, p.d.k_pool, rows, p.d.head_dim)) return false;
    if (!encode_one(enc, &p.vmap, p.d.v_pool, rows, p.d.head_dim)) return false;
    const uint64_t np = (uint64_t)p.d.num_pages;
    const int hkv = p.d.n_kv_heads, d = p.d.head_dim;
    if (!encode_run(enc, &p.kmap4, p.d.k_pool, np, hkv, d, 4) || !encode_run(enc, &p.vmap4, p.d.v_pool, np, hkv, d, 4) ||
        !encode_run(enc, &p.kmap8, p.d.k_pool, np, hkv, d, 8) || !encode_run(enc, &p.vmap8, p.d.v_pool, np, hkv, d, 8))
        return false;
    void* pair = const_cast<float4*>(p.view().rope_pair);
    p.have_rmap = p.d.max_position >= 8 * kPage && encode_rows(enc, &p.rmap, pair, p.d.max_position, d, 8) &&
                  encode_rows(enc, &p.rmap4, pair, p.d.max_position, d, 4);
    p.have_maps = true;
    return true;
}

}  // namespace lazyattn
