// Host side of the C ABI: argument validation, the pool's page allocator,
// position-table construction and kernel dispatch. See include/lazyattn.h.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <new>
#include <thread>
#include <utility>
#include <vector>

#include "internal.h"

using namespace lazyattn;

lazyattn::PoolView lazyattn_pool::view() const {
    PoolView v;
    v.k_pool = d.k_pool;
    v.v_pool = d.v_pool;
    v.rope = static_cast<const float2*>(d.rope_table);
    v.rope_pair = reinterpret_cast<const float4*>(v.rope + (size_t)d.max_position * (size_t)(d.head_dim / 2));
    v.status = d.status_word;
    v.num_pages = d.num_pages;
    v.max_position = d.max_position;
    v.hq = d.n_q_heads;
    v.hkv = d.n_kv_heads;
    v.d = d.head_dim;
    v.qk_scale = qk_scale;
    v.interleaved = d.rope_interleaved;
    return v;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launching entry points run on the pool's device only: its buffers and tensor
// maps belong to that device.
static int check_device(const lazyattn_pool* pool) {
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return LAZYATTN_ECUDA;
    return device == pool->device ? LAZYATTN_OK : LAZYATTN_EINVAL;
}

extern "C" {

const char* lazyattn_status_string(int s) {
    switch (s) {
        case LAZYATTN_OK: return "ok";
        case LAZYATTN_EINVAL: return "invalid argument";
        case LAZYATTN_ENOSPC: return "not enough free pages";
        case LAZYATTN_ERANGE: return "page id or logical position out of range";
        case LAZYATTN_EDTYPE: return "unsupported dtype for this entry point";
        case LAZYATTN_ECUDA: return "CUDA runtime error";
        case LAZYATTN_EDEVICE: return "device-side check failed";
        case LAZYATTN_EWORKSPACE: return "workspace too small";
        case LAZYATTN_ENODECODE: return "request has no writable free slot for decode";
        default: return "unknown status";
    }
}

uint64_t lazyattn_pack_entry(int32_t page, int32_t start, int32_t nvalid, int32_t writable) {
    return make_entry((uint32_t)page, start, nvalid, writable != 0);
}

size_t lazyattn_rope_table_bytes(int32_t head_dim, int32_t max_position) {
    if (head_dim <= 0 || max_position <= 0) return 0;
    return 2 * (size_t)max_position * (size_t)(head_dim / 2) * sizeof(float2);   // two layouts
}

// theta_i, i < D/2, of the pool's RoPE variant (fp64), and the logit scale.
static void rope_frequencies(const lazyattn_pool_desc& d, double* inv, float* qk_scale) {
    const int half = d.head_dim / 2;
    const double D = (double)d.head_dim, s = d.rope_factor, two_pi = 6.283185307179586476925286766559;
    double base = d.rope_theta;
    if (d.rope_scaling == LAZYATTN_ROPE_NTK) base *= pow(s, D / (D - 2.0));
    for (int i = 0; i < half; ++i) {
        const double th = pow(base, -2.0 * (double)i / D);
        double out = th;
        switch (d.rope_scaling) {
        case LAZYATTN_ROPE_LINEAR:
            out = th / s;
            break;
        case LAZYATTN_ROPE_YARN: {
            const double r = (double)d.rope_original_max_position * th / two_pi;   // rotations in the original context
            double gamma = (r - d.rope_low) / (d.rope_high - d.rope_low);
            gamma = gamma < 0.0 ? 0.0 : (gamma > 1.0 ? 1.0 : gamma);
            out = (1.0 - gamma) * th / s + gamma * th;
            break;
        }
        case LAZYATTN_ROPE_LLAMA3: {
            const double wavelen = two_pi / th;
            const double lo_wl = (double)d.rope_original_max_position / d.rope_low;
            const double hi_wl = (double)d.rope_original_max_position / d.rope_high;
            if (wavelen < hi_wl) {
                out = th;
            } else if (wavelen > lo_wl) {
                out = th / s;
            } else {
                const double smooth = ((double)d.rope_original_max_position / wavelen - d.rope_low) /
                                      (d.rope_high - d.rope_low);
                out = (1.0 - smooth) * th / s + smooth * th;
            }
            break;
        }
        default:
            break;
        }
        inv[i] = out;
    }
    if (d.rope_scaling == LAZYATTN_ROPE_YARN && s > 1.0) {
        const double t = 0.1 * log(s) + 1.0;
        *qk_scale = (float)(t * t / sqrt(D));
    }
}

int lazyattn_pool_create(const lazyattn_pool_desc* desc, void* stream, lazyattn_pool_t* out_pool) {
    if (!desc || !out_pool) return LAZYATTN_EINVAL;
    *out_pool = nullptr;
    const lazyattn_pool_desc& d = *desc;
    if (d.num_pages < 1 || d.page_size != kPage || d.n_q_heads < 1 || d.n_kv_heads < 1 ||
        d.n_q_heads % d.n_kv_heads != 0 || !(d.rope_theta > 0.0) || d.max_position < 1 ||
        d.max_position > LAZYATTN_MAX_START + kPage)
        return LAZYATTN_EINVAL;
    if (!d.k_pool || !d.v_pool || !d.rope_table || !d.status_word) return LAZYATTN_EINVAL;
    if (d.rope_scaling < LAZYATTN_ROPE_DEFAULT || d.rope_scaling > LAZYATTN_ROPE_LLAMA3) return LAZYATTN_EINVAL;
    if (d.rope_interleaved != 0 && !(d.rope_interleaved == 1 && d.dtype == LAZYATTN_BF16)) return LAZYATTN_EINVAL;
    if (d.position_encoding != LAZYATTN_POS_ROPE &&
        !(d.position_encoding == LAZYATTN_POS_ALIBI && d.dtype == LAZYATTN_BF16 && d.rope_scaling == 0 &&
          d.rope_interleaved == 0 && d.key_storage == LAZYATTN_KEYS_POSITION_FREE))
        return LAZYATTN_EINVAL;
    if (d.key_storage != LAZYATTN_KEYS_POSITION_FREE &&
        !(d.key_storage == LAZYATTN_KEYS_DOC_LOCAL && d.dtype == LAZYATTN_BF16))
        return LAZYATTN_EINVAL;
    if (d.rope_scaling != LAZYATTN_ROPE_DEFAULT && !(d.rope_factor >= 1.0)) return LAZYATTN_EINVAL;
    if ((d.rope_scaling == LAZYATTN_ROPE_YARN || d.rope_scaling == LAZYATTN_ROPE_LLAMA3) &&
        (d.rope_original_max_position < 1 || !(d.rope_low >= 0.0) || !(d.rope_high > d.rope_low)))
        return LAZYATTN_EINVAL;
    if (!aligned16(d.k_pool) || !aligned16(d.v_pool) || !aligned16(d.rope_table) ||
        (reinterpret_cast<uintptr_t>(d.status_word) & 3u))
        return LAZYATTN_EINVAL;
    if (d.dtype == LAZYATTN_F32) {
        if (d.head_dim != 64 && d.head_dim != 128) return LAZYATTN_EINVAL;
    } else if (d.dtype == LAZYATTN_BF16) {
        if (d.head_dim != 128) return LAZYATTN_EINVAL;
        if (d.n_q_heads / d.n_kv_heads > 8) return LAZYATTN_EINVAL;   // decode packs <= 8 heads per MMA
    } else {
        return LAZYATTN_EDTYPE;
    }

    lazyattn_pool* p = new (std::nothrow) lazyattn_pool();
    if (!p) return LAZYATTN_ENOSPC;
    p->d = d;
    try {   // host memory only; no exception leaves this C entry point
        p->is_free.assign((size_t)d.num_pages, 1);
        p->free_heap.resize((size_t)d.num_pages);   // never grows past this: pushes cannot reallocate
    } catch (...) {
        delete p;
        return LAZYATTN_ENOSPC;
    }
    for (int32_t i = 0; i < d.num_pages; ++i) p->free_heap[(size_t)i] = i;   // ascending: already a min-heap

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
        delete p;
        return LAZYATTN_ECUDA;
    }
    int occ = 1;
    if (d.dtype == LAZYATTN_BF16 && (decode_occupancy(&occ) != LAZYATTN_OK || prefill_init() != LAZYATTN_OK ||
                                     decode_shared_init() != LAZYATTN_OK)) {
        delete p;
        return LAZYATTN_ECUDA;
    }
    p->decode_slots = p->sm_count * std::max(occ, 1);
    if (d.dtype == LAZYATTN_BF16 && !encode_pool_maps(*p)) {
        delete p;
        return LAZYATTN_EINVAL;   // pool too large for 32-bit TMA rows, or no tensor-map support
    }

    // Position table: angle pos * theta_i in fp64, cos/sin in fp64, stored fp32;
    // theta_i from the pool's RoPE variant.
    const int half = d.head_dim / 2;
    std::vector<float2> tab;
    std::vector<double> inv;
    try {
        tab.resize(2 * (size_t)d.max_position * (size_t)half);   // (cos, sin) rows, then the paired rows
        inv.resize((size_t)half);
    } catch (...) {
        delete p;
        return LAZYATTN_ENOSPC;
    }
    p->qk_scale = (float)(1.0 / sqrt((double)d.head_dim));
    rope_frequencies(d, inv.data(), &p->qk_scale);
    auto fill_rows = [&](int32_t lo, int32_t hi) {
        for (int32_t pos = lo; pos < hi; ++pos) {
            float2* row = &tab[(size_t)pos * half];
            for (int i = 0; i < half; ++i) {
                const double a = (double)pos * inv[i];
                row[i] = make_float2((float)cos(a), (float)sin(a));
            }
            // the same row as (cos f, cos f+1, sin f, sin f+1) groups, f even
            float2* pair = &tab[((size_t)d.max_position + (size_t)pos) * half];
            for (int i = 0; i < half; i += 2) {
                pair[i] = make_float2(row[i].x, row[i + 1].x);
                pair[i + 1] = make_float2(row[i].y, row[i + 1].y);
            }
        }
    };
    // long tables (millions of positions) are filled by several host threads
    const int32_t kRowsPerThread = 1 << 16;
    const int n_threads = (int)std::min<int64_t>(std::max(1u, std::thread::hardware_concurrency()),
                                                 std::min<int64_t>(16, ((int64_t)d.max_position + kRowsPerThread - 1) /
                                                                           kRowsPerThread));
    if (n_threads <= 1) {
        fill_rows(0, d.max_position);
    } else {
        // Rows [lo, hi) per thread; rows whose thread could not be started are
        // filled here (no exception leaves this C entry point).
        std::vector<std::thread> pool_threads;
        const int64_t per = ((int64_t)d.max_position + n_threads - 1) / n_threads;
        int32_t done_upto = 0;   // rows [0, done_upto) are handed to started threads
        for (int t = 0; t < n_threads; ++t) {
            const int32_t lo = (int32_t)std::min<int64_t>((int64_t)t * per, d.max_position);
            const int32_t hi = (int32_t)std::min<int64_t>((int64_t)(t + 1) * per, d.max_position);
            try {
                pool_threads.emplace_back(fill_rows, lo, hi);
            } catch (...) {
                break;
            }
            done_upto = hi;
        }
        fill_rows(done_upto, d.max_position);
        for (auto& th : pool_threads) th.join();
    }
    cudaError_t e = cudaMemcpyAsync(d.rope_table, tab.data(), tab.size() * sizeof(float2),
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(d.status_word, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        delete p;
        return LAZYATTN_ECUDA;
    }
    *out_pool = p;
    return LAZYATTN_OK;
}

int lazyattn_pool_destroy(lazyattn_pool_t pool) {
    if (!pool) return LAZYATTN_EINVAL;
    delete pool;
    return LAZYATTN_OK;
}

int lazyattn_pool_free_count(lazyattn_pool_t pool, int32_t* out_count) {
    if (!pool || !out_count) return LAZYATTN_EINVAL;
    *out_count = (int32_t)pool->free_heap.size();
    return LAZYATTN_OK;
}

int lazyattn_alloc_pages(lazyattn_pool_t pool, int32_t n, int32_t* out_pages) {
    if (!pool || n < 0 || (n > 0 && !out_pages)) return LAZYATTN_EINVAL;
    if ((size_t)n > pool->free_heap.size()) return LAZYATTN_ENOSPC;
    for (int32_t i = 0; i < n; ++i) {
        std::pop_heap(pool->free_heap.begin(), pool->free_heap.end(), std::greater<int32_t>());
        const int32_t pg = pool->free_heap.back();
        pool->free_heap.pop_back();
        pool->is_free[(size_t)pg] = 0;
        out_pages[i] = pg;
    }
    return LAZYATTN_OK;
}

int lazyattn_free_pages(lazyattn_pool_t pool, const int32_t* pages, int32_t n) {
    if (!pool || n < 0 || (n > 0 && !pages)) return LAZYATTN_EINVAL;
    // Validate every id before changing anything: in range, taken, not repeated
    // (repeats are found by marking each id once; marks are undone on failure).
    constexpr uint8_t kMarked = 2;
    int rc = LAZYATTN_OK;
    int32_t marked = 0;
    for (; marked < n; ++marked) {
        const int32_t pg = pages[marked];
        if (pg < 0 || pg >= pool->d.num_pages) { rc = LAZYATTN_ERANGE; break; }
        if (pool->is_free[(size_t)pg]) { rc = LAZYATTN_EINVAL; break; }   // free, or repeated (marked)
        pool->is_free[(size_t)pg] = kMarked;
    }
    if (rc != LAZYATTN_OK) {
        for (int32_t i = 0; i < marked; ++i) pool->is_free[(size_t)pages[i]] = 0;
        return rc;
    }
    // O(log free) per page; the heap hands out the lowest free id first.
    for (int32_t i = 0; i < n; ++i) {
        pool->is_free[(size_t)pages[i]] = 1;
        pool->free_heap.push_back(pages[i]);
        std::push_heap(pool->free_heap.begin(), pool->free_heap.end(), std::greater<int32_t>());
    }
    return LAZYATTN_OK;
}

int lazyattn_store_doc(lazyattn_pool_t pool, const void* k, const void* v, int32_t n_tokens, void* stream,
                       int32_t* out_pages, int32_t out_cap, int32_t* out_npages) {
    if (!pool || !k || !v || !out_pages || !out_npages || n_tokens < 1) return LAZYATTN_EINVAL;
    if (!aligned16(k) || !aligned16(v)) return LAZYATTN_EINVAL;
    const int32_t np = (n_tokens + kPage - 1) / kPage;
    if (out_cap < np) return LAZYATTN_EINVAL;
    if (pool->d.key_storage == LAZYATTN_KEYS_DOC_LOCAL && n_tokens > pool->d.max_position) return LAZYATTN_EINVAL;
    int rc = check_device(pool);
    if (rc != LAZYATTN_OK) return rc;
    rc = lazyattn_alloc_pages(pool, np, out_pages);
    if (rc != LAZYATTN_OK) return rc;
    rc = launch_store_pages(*pool, k, v, n_tokens, out_pages, np, static_cast<cudaStream_t>(stream));
    if (rc != LAZYATTN_OK) {
        lazyattn_free_pages(pool, out_pages, np);
        return rc;
    }
    *out_npages = np;
    return LAZYATTN_OK;
}

// A decode plan fits a batch when it was built for its number of requests and
// the pool's head layout and key storage, and has been uploaded.
static bool plan_fits(const lazyattn_pool* pool, const lazyattn_batch* b) {
    const lazyattn_plan* pl = b->decode_plan;
    return pl->num_requests == b->num_requests && pl->hkv == pool->d.n_kv_heads &&
           pl->g == pool->d.n_q_heads / pool->d.n_kv_heads && pl->key_storage == pool->d.key_storage &&
           pl->device != nullptr;
}

static int check_batch(const lazyattn_pool* pool, const lazyattn_batch* b, int op) {
    if (!pool || !b) return LAZYATTN_EINVAL;
    if (b->num_requests < 1 || b->num_requests > 65535 || b->max_entries < 0 || !b->entries || !b->entry_offsets)
        return LAZYATTN_EINVAL;
    if (b->flags & ~LAZYATTN_KEYS_PREROTATED) return LAZYATTN_EINVAL;
    if (pool->d.key_storage == LAZYATTN_KEYS_DOC_LOCAL &&
        ((b->flags & LAZYATTN_KEYS_PREROTATED) || (b->max_entries > 0 && !b->entry_delta)))
        return LAZYATTN_EINVAL;
    if (pool->d.position_encoding == LAZYATTN_POS_ALIBI && (b->flags & LAZYATTN_KEYS_PREROTATED)) return LAZYATTN_EINVAL;
    if (op == LAZYATTN_OP_PREFILL) {
        if (b->total_q < 0 || b->max_q_len < 0 || !b->q_offsets || !b->q_start) return LAZYATTN_EINVAL;
    }
    if (op == LAZYATTN_OP_DECODE && b->decode_plan && pool->d.dtype == LAZYATTN_BF16 && !plan_fits(pool, b))
        return LAZYATTN_EINVAL;
    return LAZYATTN_OK;
}

size_t lazyattn_workspace_size(lazyattn_pool_t pool, int32_t op, const lazyattn_batch* batch) {
    if (check_batch(pool, batch, op) != LAZYATTN_OK) return 0;
    if (op == LAZYATTN_OP_PREFILL) {
        const int splits = pool->d.dtype == LAZYATTN_BF16 ? prefill_splits(*pool, *batch) : 1;
        return splits > 1 ? prefill_ws_bytes(*pool, *batch, splits) : 256;
    }
    if (op != LAZYATTN_OP_DECODE) return 0;
    if (pool->d.dtype == LAZYATTN_F32) return (size_t)batch->num_requests * sizeof(int32_t) + 256;
    if (batch->decode_plan) return decode_plan_ws_bytes(*pool, *batch->decode_plan);
    return decode_ws_layout(*pool, *batch).total;
}

int lazyattn_prefill(lazyattn_pool_t pool, const lazyattn_batch* batch, const void* q, void* out,
                     void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_batch(pool, batch, LAZYATTN_OP_PREFILL);
    if (rc != LAZYATTN_OK) return rc;
    if (batch->total_q == 0) return LAZYATTN_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return LAZYATTN_EINVAL;
    rc = check_device(pool);
    if (rc != LAZYATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (pool->d.dtype == LAZYATTN_F32)
        return launch_attention_f32(*pool, *batch, static_cast<const float*>(q), static_cast<float*>(out),
                                    nullptr, st);
    return launch_prefill_bf16(*pool, *batch, static_cast<const __nv_bfloat16*>(q),
                               static_cast<__nv_bfloat16*>(out), workspace, workspace_bytes, st);
}

int lazyattn_decode(lazyattn_pool_t pool, const lazyattn_batch* batch, const void* q, const void* k_new,
                    const void* v_new, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_batch(pool, batch, LAZYATTN_OP_DECODE);
    if (rc != LAZYATTN_OK) return rc;
    if (!q || !k_new || !v_new || !out || !workspace) return LAZYATTN_EINVAL;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return LAZYATTN_EINVAL;
    if (workspace_bytes < lazyattn_workspace_size(pool, LAZYATTN_OP_DECODE, batch)) return LAZYATTN_EWORKSPACE;
    rc = check_device(pool);
    if (rc != LAZYATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (pool->d.dtype == LAZYATTN_F32) {
        int32_t* qpos = static_cast<int32_t*>(workspace);
        rc = launch_decode_append(*pool, *batch, k_new, v_new, qpos, st);
        if (rc != LAZYATTN_OK) return rc;
        return launch_attention_f32(*pool, *batch, static_cast<const float*>(q), static_cast<float*>(out),
                                    qpos, st);
    }
    if (batch->decode_plan) {   // document-major: qpos at the workspace's start, then the partials
        rc = launch_decode_append(*pool, *batch, k_new, v_new, static_cast<int32_t*>(workspace), st);
        if (rc != LAZYATTN_OK) return rc;
        return launch_decode_shared(*pool, *batch, *batch->decode_plan, static_cast<const __nv_bfloat16*>(q),
                                    static_cast<__nv_bfloat16*>(out), workspace, st);
    }
    const DecodeWs L = decode_ws_layout(*pool, *batch);
    int32_t* qpos = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + L.qpos_off);
    rc = launch_decode_append(*pool, *batch, k_new, v_new, qpos, st);
    if (rc != LAZYATTN_OK) return rc;
    return launch_decode_bf16(*pool, *batch, static_cast<const __nv_bfloat16*>(q),
                              static_cast<__nv_bfloat16*>(out), workspace, L, st);
}

int lazyattn_materialize(lazyattn_pool_t pool, const lazyattn_batch* batch, const uint64_t* dst_entries,
                         void* stream) {
    int rc = check_batch(pool, batch, LAZYATTN_OP_DECODE);
    if (rc != LAZYATTN_OK) return rc;
    if (!dst_entries || (batch->flags & LAZYATTN_KEYS_PREROTATED) ||
        pool->d.key_storage == LAZYATTN_KEYS_DOC_LOCAL || pool->d.position_encoding == LAZYATTN_POS_ALIBI)
        return LAZYATTN_EINVAL;
    if (batch->max_entries == 0) return LAZYATTN_OK;
    rc = check_device(pool);
    if (rc != LAZYATTN_OK) return rc;
    return launch_materialize(*pool, *batch, dst_entries, static_cast<cudaStream_t>(stream));
}

int lazyattn_resolve(lazyattn_pool_t pool, const lazyattn_batch* batch, const int32_t* out_offsets,
                     int32_t* out_triples, int32_t out_cap, void* stream) {
    int rc = check_batch(pool, batch, LAZYATTN_OP_DECODE);
    if (rc != LAZYATTN_OK) return rc;
    if (!out_offsets || !out_triples || out_cap < 0) return LAZYATTN_EINVAL;
    rc = check_device(pool);
    if (rc != LAZYATTN_OK) return rc;
    return launch_resolve(*pool, *batch, out_offsets, out_triples, out_cap, static_cast<cudaStream_t>(stream));
}

int lazyattn_check_batch_host(const uint64_t* entries, const int32_t* entry_offsets, int32_t num_requests,
                              int32_t num_pages, int32_t max_position, int32_t* out_request) {
    if (out_request) *out_request = -1;
    if (!entry_offsets || num_requests < 0 || num_pages < 1 || max_position < 1) return LAZYATTN_EINVAL;
    if (num_requests > 0 && entry_offsets[0] < 0) return LAZYATTN_EINVAL;
    for (int32_t r = 0; r < num_requests; ++r)
        if (entry_offsets[r + 1] < entry_offsets[r]) return LAZYATTN_EINVAL;
    if (num_requests > 0 && entry_offsets[num_requests] > 0 && !entries) return LAZYATTN_EINVAL;
    std::vector<std::pair<int64_t, int64_t>> spans;   // [start, start + nvalid) of one request
    for (int32_t r = 0; r < num_requests; ++r) {
        int rc = LAZYATTN_OK;
        try {
            spans.clear();
            for (int32_t i = entry_offsets[r]; i < entry_offsets[r + 1]; ++i) {
                const uint64_t e = entries[i];
                const int32_t n = entry_nvalid(e);
                if (n == 0) continue;
                if (entry_page(e) >= (uint32_t)num_pages || n > kPage || entry_start(e) + n > max_position) {
                    rc = LAZYATTN_ERANGE;
                    break;
                }
                spans.emplace_back(entry_start(e), entry_start(e) + n);
            }
        } catch (...) {
            return LAZYATTN_ENOSPC;
        }
        if (rc == LAZYATTN_OK) {
            std::sort(spans.begin(), spans.end());
            for (size_t i = 1; i < spans.size(); ++i)
                if (spans[i].first < spans[i - 1].second) {
                    rc = LAZYATTN_EINVAL;
                    break;
                }
        }
        if (rc != LAZYATTN_OK) {
            if (out_request) *out_request = r;
            return rc;
        }
    }
    return LAZYATTN_OK;
}

int lazyattn_get_device_status(lazyattn_pool_t pool, int32_t* out_status, int32_t reset, void* stream) {
    if (!pool || !out_status) return LAZYATTN_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, pool->d.status_word, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && reset) e = cudaMemsetAsync(pool->d.status_word, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return LAZYATTN_ECUDA;
    *out_status = h;
    return LAZYATTN_OK;
}

}  // extern "C"
