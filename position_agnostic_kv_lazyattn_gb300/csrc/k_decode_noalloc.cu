// lazyattn_decode_noalloc: the decode step for callers that cannot allocate
// device memory.
//
// lazyattn_decode needs a caller-provided workspace (the appended tokens'
// positions, the split-combine tickets and the per-split partial results).
// Some callers have no way to obtain one: code running where cudaMalloc is
// forbidden or unavailable (inside an allocator-less runtime, a plugin whose
// host owns all device memory, or a context that must not grow its footprint
// after start-up). For them this entry point uses a fixed scratch array that
// lives in the library itself, in device global memory, sized for a stated
// maximum; it allocates nothing.
#include <mutex>

#include "internal.h"

namespace {

// One copy per GPU that loads the library, held until the process exits.
__device__ __align__(256) unsigned char g_decode_scratch[LAZYATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
// The host-side symbol is only a stand-in; the real address has to be asked
// for once per device.
int scratch_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return LAZYATTN_EINVAL;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return LAZYATTN_ECUDA;
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return LAZYATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int lazyattn_decode_noalloc(lazyattn_pool_t pool, const lazyattn_batch* batch_in, const void* q,
                                       const void* k_new, const void* v_new, void* out, void* stream) {
    using namespace lazyattn;
    if (!pool || !batch_in) return LAZYATTN_EINVAL;
    lazyattn_batch batch_copy = *batch_in;
    batch_copy.decode_plan = nullptr;   // each request reads its own pages (a plan's image needs device memory)
    const lazyattn_batch* batch = &batch_copy;
    const size_t need = lazyattn_workspace_size(pool, LAZYATTN_OP_DECODE, batch);   // 0: invalid batch
    if (need == 0) return LAZYATTN_EINVAL;
    if (need > (size_t)LAZYATTN_NOALLOC_SCRATCH_BYTES) return LAZYATTN_EWORKSPACE;
    if (!q || !k_new || !v_new || !out || !aligned16(q) || !aligned16(k_new) || !aligned16(v_new) ||
        !aligned16(out))
        return LAZYATTN_EINVAL;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return LAZYATTN_ECUDA;
    if (device != pool->device) return LAZYATTN_EINVAL;
    void* scratch = nullptr;
    int rc = scratch_address(device, &scratch);
    if (rc != LAZYATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (pool->d.dtype == LAZYATTN_F32) {
        int32_t* qpos = static_cast<int32_t*>(scratch);   // written by the append kernel before it is read
        rc = launch_decode_append(*pool, *batch, k_new, v_new, qpos, st);
        if (rc != LAZYATTN_OK) return rc;
        return launch_attention_f32(*pool, *batch, static_cast<const float*>(q), static_cast<float*>(out), qpos, st);
    }
    const DecodeWs L = decode_ws_layout(*pool, *batch);
    char* base = static_cast<char*>(scratch);
    // The array keeps whatever the previous call left; the split-combine
    // tickets must start at zero.
    const size_t ticket_bytes = (size_t)batch->num_requests * (size_t)pool->d.n_kv_heads * sizeof(int32_t);
    if (cudaMemsetAsync(base + L.ticket_off, 0, ticket_bytes, st) != cudaSuccess) return LAZYATTN_ECUDA;
    int32_t* qpos = reinterpret_cast<int32_t*>(base + L.qpos_off);
    rc = launch_decode_append(*pool, *batch, k_new, v_new, qpos, st);
    if (rc != LAZYATTN_OK) return rc;
    return launch_decode_bf16(*pool, *batch, static_cast<const __nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(out),
                              scratch, L, st);
}
