// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <vector>

#include "lazyattn.h"

namespace lazyattn {

constexpr int kPage = LAZYATTN_PAGE_SIZE;

// ---------------------------------------------------------------- entries
// Field layout fixed by lazyattn_pack_entry (lazyattn.h).
__host__ __device__ __forceinline__ uint32_t entry_page(uint64_t e) { return (uint32_t)(e & 0xffffffffull); }
__host__ __device__ __forceinline__ int32_t entry_start(uint64_t e) { return (int32_t)((e >> 32) & ((1ull << 26) - 1)); }
__host__ __device__ __forceinline__ int32_t entry_nvalid(uint64_t e) { return (int32_t)((e >> 58) & 0x1f); }
__host__ __device__ __forceinline__ bool entry_writable(uint64_t e) { return (e >> 63) != 0; }
__host__ __device__ __forceinline__ uint64_t make_entry(uint32_t page, int32_t start, int32_t nvalid, bool w) {
    return (uint64_t)page | ((uint64_t)(start & ((1 << 26) - 1)) << 32) | ((uint64_t)(nvalid & 0x1f) << 58) |
           ((uint64_t)(w ? 1 : 0) << 63);
}

// ---------------------------------------------------------------- dependent launches
// Programmatic dependent launch: a kernel launched with launch_dependent may
// start while the previous kernel in the stream still runs. It must call
// grid_dep_wait() before reading anything that kernel writes; the wait
// returns once the previous grid has completed and its writes are visible
// (and at once when there is no such dependency). grid_dep_launch_dependents()
// lets the next such launch start early.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Shape and buffers a kernel needs about the pool (passed by value).
struct PoolView {
    void* k_pool;
    void* v_pool;
    const float2* rope;   // [max_position][D/2] (cos, sin)
    const float4* rope_pair;   // [max_position][D/4] (cos f, cos f+1, sin f, sin f+1), f even
    int32_t* status;
    int32_t num_pages;
    int32_t max_position;
    int32_t hq, hkv, d;
    float qk_scale;       // logit scale: 1/sqrt(D), times YaRN's attention temperature
    int32_t interleaved;  // q/k arrive with interleaved RoPE pairs (2i, 2i+1): de-interleave on load
};

// ALiBi slope of query head h out of n (the ALiBi paper's rule): for n a power
// of two, 2^(-8 (h+1) / n); otherwise the slopes of p = the power of two below
// n for h < p, then every other slope of 2p (its 1st, 3rd, ...) for h >= p.
__host__ __device__ inline float alibi_slope(int h, int n) {
    int p = 1;
    while (p * 2 <= n) p *= 2;
    if (h < p) return exp2f(-8.0f * (float)(h + 1) / (float)p);
    return exp2f(-8.0f * (float)(2 * (h - p) + 1) / (float)(2 * p));
}

// Interleaved RoPE pairs: from 16 consecutive bf16 of a q or k row (two uint4,
// elements 16u .. 16u+15), the 8 even elements (pair members 2i, which become
// dims 8u.. of the first half) and the 8 odd ones (dims 64+8u.. of the second).
// (Safe when even / odd alias a / b: both results are formed before either is written.)
__device__ __forceinline__ void deinterleave16(const uint4& a, const uint4& b, uint4& even, uint4& odd) {
    const uint4 e = make_uint4(__byte_perm(a.x, a.y, 0x5410), __byte_perm(a.z, a.w, 0x5410),
                               __byte_perm(b.x, b.y, 0x5410), __byte_perm(b.z, b.w, 0x5410));
    const uint4 o = make_uint4(__byte_perm(a.x, a.y, 0x7632), __byte_perm(a.z, a.w, 0x7632),
                               __byte_perm(b.x, b.y, 0x7632), __byte_perm(b.z, b.w, 0x7632));
    even = e;
    odd = o;
}

// Record the first device-side error; later ones are dropped.
__device__ __forceinline__ void record_error(int32_t* status, int32_t code) {
    atomicCAS(status, 0, code);
}

// Input range of the bf16 kernels (lazyattn.h, "Input range"). Their QK^T MMAs
// take fp16 operands: a key rotated at any angle, and q rotated and scaled by
// log2(e) times the logit scale. A rotation keeps the norm of each rotate-half
// pair (x_i, x_{i+D/2}). With the norm at most 65024 a pair stays finite in
// fp16 on every path: rotated once (<= 65024); rotated and stored as bf16 (the
// materialised baseline: each component rounds to at most 65280); or stored
// rotated as bf16 at document-local positions (the rounding grows the norm by
// at most 2^-8, to 65278) and rotated again by the document's offset; fp16's
// largest value is 65504. Checked in fp32 on the values as they arrive; a
// violation is recorded as LAZYATTN_ERANGE.
constexpr float kMaxPairNorm = 65024.0f;
constexpr float kMaxPairNorm2 = kMaxPairNorm * kMaxPairNorm;

// Largest squared pair norm of 8 rotate-half pairs: bf16 x8 of the first half
// (a) and of the second half (b).
__device__ __forceinline__ float max_pair_norm2(const uint4& a, const uint4& b) {
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = __uint_as_float(av[i] << 16), x1 = __uint_as_float(av[i] & 0xffff0000u);
        const float y0 = __uint_as_float(bv[i] << 16), y1 = __uint_as_float(bv[i] & 0xffff0000u);
        m = fmaxf(m, fmaxf(fmaf(x0, x0, y0 * y0), fmaf(x1, x1, y1 * y1)));
        if (!(x0 == x0 && x1 == x1 && y0 == y0 && y1 == y1)) m = INFINITY;   // NaN: out of range too
    }
    return m;
}

// An entry is usable iff its page and every position it covers are in range.
// Entries failing the check are skipped and reported.
__device__ __forceinline__ bool entry_ok(const PoolView& pv, uint64_t e) {
    const int32_t n = entry_nvalid(e);
    if (n == 0) return true;
    if (entry_page(e) >= (uint32_t)pv.num_pages || n > kPage ||
        entry_start(e) + n > pv.max_position) {
        record_error(pv.status, LAZYATTN_ERANGE);
        return false;
    }
    return true;
}

// Decode workspace layout (byte offsets from the workspace base).
struct DecodeWs {
    size_t qpos_off;      // int32 [R]: logical position of the appended token
    size_t ticket_off;    // int32 [R*Hkv]: split-combine tickets (zero at rest)
    size_t ml_off;        // float2 [R*Hkv*S][g]: (m, l) of each split, log2 domain
    size_t acc_off;       // float [R*Hkv*S][g][D]: unnormalised partial outputs
    size_t total;
    int splits;
};

// ---------------------------------------------------------------- decode plan
// Device image of a decode plan (lazyattn_decode_plan_create): work units,
// their users and each request's range of partial results.
struct PlanUnit {
    int32_t entry0;    // batch entry of the unit's first page in its first user's table
    int32_t n_pages;   // pages (entries) of the unit
    int32_t user0;     // first user of the unit in the users array
    int32_t n_users;   // users of the unit (bit 31: private tail run, read after the append)
};
constexpr int32_t kUnitPrivate = int32_t(1u << 31);
struct PlanUser {
    int32_t request;
    int32_t delta;     // logical position of the unit's run-local position 0 in this request
    int32_t partial;   // partial-result slot of (this user, this unit)
    int32_t pad;
};

}  // namespace lazyattn

struct lazyattn_plan {
    int32_t num_requests = 0;
    int32_t num_units = 0;
    int32_t num_users = 0;
    int32_t num_partials = 0;
    int32_t g = 0, hkv = 0;
    int32_t key_storage = 0;
    size_t units_off = 0, users_off = 0, pbase_off = 0;
    std::vector<uint8_t> image;        // the device image, uploaded by lazyattn_decode_plan_upload
    void* device = nullptr;            // where it was uploaded (caller-owned)
    lazyattn_decode_plan_stats stats{};
};

struct lazyattn_pool {
    lazyattn_pool_desc d;
    std::vector<int32_t> free_heap;    // free page ids, a min-heap (std::greater): lowest id first
    std::vector<uint8_t> is_free;
    int device = 0;
    int sm_count = 0;
    int decode_slots = 0;              // resident decode CTAs on the whole GPU
    float qk_scale = 0.f;              // logit scale (1/sqrt(D), YaRN temperature included)
    bool have_maps = false;            // bf16 pools: TMA views of the K and V pools
    CUtensorMap kmap, vmap;            // rows of 128 dims, boxes of one page (64 dims x 16 slots)
    CUtensorMap kmap4, vmap4;          // {D, slot, KV head, page}, boxes of four consecutive pages
    CUtensorMap kmap8, vmap8;          // the same view, boxes of eight consecutive pages
    bool have_rmap = false;            // rmap encoded (position tables of at least 128 rows)
    CUtensorMap rmap, rmap4;           // paired position table as {D floats, 16, max_position / 16}:
                                       // a box holds rows p, p + 16, ..., p + 112 (eight pages' starts;
                                       // rmap4: four pages')
    lazyattn::PoolView view() const;
};

namespace lazyattn {

// ---------------------------------------------------------------- launchers
// Each returns a lazyattn_status; all enqueue on `stream` and never block.
int launch_store_pages(const lazyattn_pool& p, const void* k, const void* v, int32_t n_tokens,
                       const int32_t* pages_host, int32_t npages, cudaStream_t stream);
int launch_decode_append(const lazyattn_pool& p, const lazyattn_batch& b, const void* k_new,
                         const void* v_new, int32_t* qpos, cudaStream_t stream);
int launch_materialize(const lazyattn_pool& p, const lazyattn_batch& b, const uint64_t* dst,
                       cudaStream_t stream);
int launch_resolve(const lazyattn_pool& p, const lazyattn_batch& b, const int32_t* out_offsets,
                   int32_t* out, int32_t cap, cudaStream_t stream);

// TMA views of the bf16 K and V pools as rows of 128 elements (row = (page *
// Hkv + kv head) * 16 + slot), 64 x 16 boxes, and as 4-D {D, slot, KV head,
// page} tensors with boxes of four consecutive pages; 128-byte swizzle. False
// if the driver entry point is unavailable or the pool is too large for
// 32-bit rows.
bool encode_pool_maps(lazyattn_pool& p);

// fp32 SIMT attention (prefill rows or one decode row per request).
int launch_attention_f32(const lazyattn_pool& p, const lazyattn_batch& b, const float* q, float* out,
                         const int32_t* decode_qpos, cudaStream_t stream);

// bf16 decode: split-K over pages, tensor-core dot products (mma.sync), RoPE in registers.
DecodeWs decode_ws_layout(const lazyattn_pool& p, const lazyattn_batch& b);
int decode_occupancy(int* ctas_per_sm);
int launch_decode_bf16(const lazyattn_pool& p, const lazyattn_batch& b, const __nv_bfloat16* q,
                       __nv_bfloat16* out, void* ws, const DecodeWs& L, cudaStream_t stream);

// bf16 decode through a plan: document-major units on tcgen05 / TMEM, then a
// combine of each request's partial results.
size_t decode_plan_ws_bytes(const lazyattn_pool& p, const lazyattn_plan& plan);
int decode_shared_init();
int launch_decode_shared(const lazyattn_pool& p, const lazyattn_batch& b, const lazyattn_plan& plan,
                         const __nv_bfloat16* q, __nv_bfloat16* out, void* ws, cudaStream_t stream);

// bf16 prefill on tcgen05 / TMEM with TMA-staged K/V tiles. prefill_init()
// sets the kernel's shared-memory limit on the current device (done once, at
// pool creation, so that launches stay capturable in CUDA graphs).
int prefill_init();
// Split count of a bf16 prefill over the KV tiles (1: one CTA per request, KV
// head and query pair) and the workspace bytes its partials take.
int prefill_splits(const lazyattn_pool& p, const lazyattn_batch& b);
size_t prefill_ws_bytes(const lazyattn_pool& p, const lazyattn_batch& b, int splits);
int launch_prefill_bf16(const lazyattn_pool& p, const lazyattn_batch& b, const __nv_bfloat16* q,
                        __nv_bfloat16* out, void* ws, size_t ws_bytes, cudaStream_t stream);

}  // namespace lazyattn
