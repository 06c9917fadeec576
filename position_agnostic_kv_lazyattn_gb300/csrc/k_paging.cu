// Page-level kernels: storing pre-RoPE K/V into pages, the decode-step append,
// the materialising baseline's copy-and-rotate, and the debug table resolver.
#include "internal.h"

namespace lazyattn {

namespace {

constexpr int kMaxPagesPerLaunch = 512;

struct PageList {
    int32_t ids[kMaxPagesPerLaunch];
};

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// src [n_tokens][Hkv][D] -> pages [page][Hkv][16][D]; one block per (page, kv head).
// Slots past n_tokens in the last page are zero-filled.
// interleaved (bf16): K rows are de-interleaved on the way (pairs (2i, 2i+1) of
// an interleaved-RoPE model become the rotate-half pairs (i, i + D/2)).
// check_range (bf16 pools): every stored key pair must satisfy the input range
// of the bf16 kernels (max_pair_norm2); a violation is recorded in status.
__global__ void store_pages_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* kp, uint4* vp,
                                   int32_t n_tokens, int32_t first_page_index, PageList pages, int hkv,
                                   int row_vecs, int interleaved, int check_range, int32_t* status) {
    const int j = blockIdx.x;          // page index within this launch
    const int h = blockIdx.y;
    const int32_t page = pages.ids[j];
    const int tok0 = (first_page_index + j) * kPage;
    const size_t dst_base = ((size_t)page * hkv + h) * kPage * row_vecs;
    if (interleaved) {
        const int hv = row_vecs / 2;
        for (int i = threadIdx.x; i < kPage * hv; i += blockDim.x) {
            const int slot = i / hv, u = i % hv;
            const int tok = tok0 + slot;
            uint4 ev = make_uint4(0, 0, 0, 0), od = ev;
            if (tok < n_tokens) {
                const size_t src = ((size_t)tok * hkv + h) * row_vecs + 2 * u;
                deinterleave16(k[src], k[src + 1], ev, od);
                if (check_range && max_pair_norm2(ev, od) > kMaxPairNorm2) record_error(status, LAZYATTN_ERANGE);
            }
            kp[dst_base + (size_t)slot * row_vecs + u] = ev;
            kp[dst_base + (size_t)slot * row_vecs + hv + u] = od;
        }
        for (int i = threadIdx.x; i < kPage * row_vecs; i += blockDim.x) {
            const int slot = i / row_vecs, c = i % row_vecs;
            const int tok = tok0 + slot;
            vp[dst_base + i] = tok < n_tokens ? v[((size_t)tok * hkv + h) * row_vecs + c] : make_uint4(0, 0, 0, 0);
        }
        return;
    }
    for (int i = threadIdx.x; i < kPage * row_vecs; i += blockDim.x) {
        const int slot = i / row_vecs, c = i % row_vecs;
        const int tok = tok0 + slot;
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (tok < n_tokens) {
            const size_t src = ((size_t)tok * hkv + h) * row_vecs + c;
            a = k[src];
            b = v[src];
            // pairs (dims of vector c, dims of vector c + row_vecs / 2)
            if (check_range && c < row_vecs / 2 && max_pair_norm2(a, k[src + row_vecs / 2]) > kMaxPairNorm2)
                record_error(status, LAZYATTN_ERANGE);
        }
        kp[dst_base + i] = a;
        vp[dst_base + i] = b;
    }
}

// Doc-local pools (bf16): as store_pages_kernel, with K rotated at the token's
// position within the stored run (its document-local position, §3.2: a
// document's cache is encoded from position 0). Thread = (slot, 8 dims of the
// first half) and their rotate-half partners.
__global__ void store_pages_local_kernel(const __nv_bfloat16* __restrict__ k, const uint4* __restrict__ v,
                                         __nv_bfloat16* kp, uint4* vp, const float2* rope, int32_t n_tokens,
                                         int32_t first_page_index, PageList pages, int hkv, int D, int interleaved,
                                         int32_t* status) {
    const int j = blockIdx.x, h = blockIdx.y;
    const int32_t page = pages.ids[j];
    const int tok0 = (first_page_index + j) * kPage;
    const int half = D / 2, g8 = half / 8, row_vecs = D / 8;
    const size_t dst_rows = ((size_t)page * hkv + h) * kPage;
    for (int i = threadIdx.x; i < kPage * g8; i += blockDim.x) {
        const int slot = i / g8, d = (i % g8) * 8;
        const int tok = tok0 + slot;
        __nv_bfloat16* krow = kp + (dst_rows + slot) * D;
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (tok < n_tokens) {
            const __nv_bfloat16* src = k + ((size_t)tok * hkv + h) * D;
            __nv_bfloat16 x[8], y[8];
            if (interleaved) {
                uint4 ev, od;
                deinterleave16(*reinterpret_cast<const uint4*>(src + 2 * d), *reinterpret_cast<const uint4*>(src + 2 * d + 8),
                               ev, od);
                *reinterpret_cast<uint4*>(x) = ev;
                *reinterpret_cast<uint4*>(y) = od;
            } else {
                *reinterpret_cast<uint4*>(x) = *reinterpret_cast<const uint4*>(src + d);
                *reinterpret_cast<uint4*>(y) = *reinterpret_cast<const uint4*>(src + d + half);
            }
            if (max_pair_norm2(*reinterpret_cast<const uint4*>(x), *reinterpret_cast<const uint4*>(y)) > kMaxPairNorm2)
                record_error(status, LAZYATTN_ERANGE);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float2 cs = rope[(size_t)tok * half + d + t];
                const float p = __bfloat162float(x[t]), q = __bfloat162float(y[t]);
                x[t] = __float2bfloat16_rn(p * cs.x - q * cs.y);
                y[t] = __float2bfloat16_rn(p * cs.y + q * cs.x);
            }
            a = *reinterpret_cast<uint4*>(x);
            b = *reinterpret_cast<uint4*>(y);
        }
        *reinterpret_cast<uint4*>(krow + d) = a;
        *reinterpret_cast<uint4*>(krow + d + half) = b;
    }
    for (int i = threadIdx.x; i < kPage * row_vecs; i += blockDim.x) {
        const int slot = i / row_vecs, c = i % row_vecs;
        const int tok = tok0 + slot;
        vp[(dst_rows + slot) * row_vecs + c] = tok < n_tokens ? v[((size_t)tok * hkv + h) * row_vecs + c]
                                                                : make_uint4(0, 0, 0, 0);
    }
}

// Find the append slot of request r: the first entry with nvalid < 16 in the
// trailing run of writable entries. One warp scans 32 entries per step from
// the end of the request's entries. Returns the entry index or -1 (all lanes).
__device__ int find_append_entry(const uint64_t* entries, int e0, int e1, int lane) {
    int tail = -1;
    for (int base = e1 - 1; base >= e0; base -= 32) {
        const int i = base - lane;
        const bool in = i >= e0;
        const uint64_t e = in ? entries[i] : 0ull;
        const bool w = in && entry_writable(e);
        const unsigned brk = __ballot_sync(0xffffffffu, !w);            // run ends at the first such lane
        const int stop = brk ? __ffs(brk) - 1 : 32;
        unsigned cand = __ballot_sync(0xffffffffu, w && entry_nvalid(e) < kPage);
        if (stop < 32) cand &= (1u << stop) - 1u;
        if (cand) tail = base - (31 - __clz(cand));                     // furthest back = first in table order
        if (stop < 32) break;
    }
    return tail;
}

// One block per request: append k_new/v_new into the request's tail page.
// Launched as a programmatic dependent of the previous kernel in the stream
// (the previous step's attention): it lets its own dependent launch at once
// and waits for the previous grid before touching the table or the pool.
// MODE: 0 stores k as given (position-free keys); 1 rotates it at its logical
// position (pre-rotated pages of the materialising baseline); 2 at its
// document-local position, logical - entry_delta (doc-local pools).
template <typename T, int MODE>
__global__ void decode_append_kernel(PoolView pv, uint64_t* entries, const int32_t* entry_offsets,
                                     const T* __restrict__ k_new, const T* __restrict__ v_new, int32_t* qpos,
                                     const int32_t* entry_delta) {
    constexpr bool PREROT = MODE != 0;
    const int r = blockIdx.x;
    __shared__ int s_entry;
    __shared__ uint64_t s_e;
    grid_dep_launch_dependents();
    grid_dep_wait();
    if (threadIdx.x < 32) {
        const int e0 = entry_offsets[r], e1 = entry_offsets[r + 1];
        int t = find_append_entry(entries, e0, e1, threadIdx.x);
        if (threadIdx.x == 0) {
            if (t >= 0) {
                const uint64_t e = entries[t];
                const int32_t pos = entry_start(e) + entry_nvalid(e);
                if (entry_page(e) >= (uint32_t)pv.num_pages || pos >= pv.max_position) {
                    record_error(pv.status, LAZYATTN_ERANGE);
                    t = -1;
                }
            } else {
                record_error(pv.status, LAZYATTN_ENODECODE);
            }
            s_entry = t;
            s_e = t >= 0 ? entries[t] : 0;
            qpos[r] = t >= 0 ? entry_start(s_e) + entry_nvalid(s_e) : -1;
        }
    }
    __syncthreads();
    if (s_entry < 0) return;
    const uint64_t e = s_e;
    const uint32_t page = entry_page(e);
    const int slot = entry_nvalid(e);
    int pos = entry_start(e) + slot;
    if (MODE == 2) {   // rotate at the local position instead
        const int delta = entry_delta[s_entry];
        if (delta < 0 || delta > entry_start(e)) {
            if (threadIdx.x == 0) record_error(pv.status, LAZYATTN_ERANGE);
            return;
        }
        pos -= delta;
    }
    const int D = pv.d, half = D / 2;
    T* kp = static_cast<T*>(pv.k_pool);
    T* vp = static_cast<T*>(pv.v_pool);
    if (slot == 0) {
        // The first token into a page: its other slots (whatever the page held
        // before) become zeros, so that slots past a page's valid count are
        // zero in every page the library fills (the attention kernels read
        // whole pages and only mask the scores of empty slots).
        const int row = D * (int)sizeof(T) / 16;   // 16-byte vectors per row
        uint4* k4 = reinterpret_cast<uint4*>(kp);
        uint4* v4 = reinterpret_cast<uint4*>(vp);
        for (int i = threadIdx.x; i < pv.hkv * (kPage - 1) * row; i += blockDim.x) {
            const int h = i / ((kPage - 1) * row), rest = i % ((kPage - 1) * row);
            const size_t at = ((((size_t)page * pv.hkv + h) * kPage) + 1) * row + rest;
            k4[at] = make_uint4(0, 0, 0, 0);
            v4[at] = make_uint4(0, 0, 0, 0);
        }
    }
    if (sizeof(T) == 2 && half % 8 == 0) {
        // 16-byte vectors: thread = (kv head, 8 dims of the first half) and
        // their rotate-half partners; rows are 16-byte aligned (D % 16 == 0,
        // aligned k_new / v_new / pools)
        const int g8 = half / 8;
        for (int i = threadIdx.x; i < pv.hkv * g8; i += blockDim.x) {
            const int h = i / g8, d = (i % g8) * 8;
            const size_t src = ((size_t)r * pv.hkv + h) * D;
            const size_t dst = (((size_t)page * pv.hkv + h) * kPage + slot) * D;
            uint4 k1, k2;
            if (pv.interleaved) {
                deinterleave16(*reinterpret_cast<const uint4*>(k_new + src + 2 * d),
                               *reinterpret_cast<const uint4*>(k_new + src + 2 * d + 8), k1, k2);
            } else {
                k1 = *reinterpret_cast<const uint4*>(k_new + src + d);
                k2 = *reinterpret_cast<const uint4*>(k_new + src + d + half);
            }
            const uint4 v1 = *reinterpret_cast<const uint4*>(v_new + src + d);
            const uint4 v2 = *reinterpret_cast<const uint4*>(v_new + src + d + half);
            if (max_pair_norm2(k1, k2) > kMaxPairNorm2) record_error(pv.status, LAZYATTN_ERANGE);
            if (PREROT) {
                T a[8], b[8];
                *reinterpret_cast<uint4*>(a) = k1;
                *reinterpret_cast<uint4*>(b) = k2;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 cs = pv.rope[(size_t)pos * half + d + j];
                    const float x = to_f(a[j]), y = to_f(b[j]);
                    a[j] = from_f<T>(x * cs.x - y * cs.y);
                    b[j] = from_f<T>(x * cs.y + y * cs.x);
                }
                k1 = *reinterpret_cast<const uint4*>(a);
                k2 = *reinterpret_cast<const uint4*>(b);
            }
            *reinterpret_cast<uint4*>(kp + dst + d) = k1;
            *reinterpret_cast<uint4*>(kp + dst + d + half) = k2;
            *reinterpret_cast<uint4*>(vp + dst + d) = v1;
            *reinterpret_cast<uint4*>(vp + dst + d + half) = v2;
        }
    } else
    for (int i = threadIdx.x; i < pv.hkv * half; i += blockDim.x) {
        const int h = i / half, d = i % half;
        const size_t src = ((size_t)r * pv.hkv + h) * D;
        const size_t dst = (((size_t)page * pv.hkv + h) * kPage + slot) * D;
        float k1 = to_f(k_new[src + d]), k2 = to_f(k_new[src + d + half]);
        if (PREROT) {
            const float2 cs = pv.rope[(size_t)pos * half + d];
            const float a = k1 * cs.x - k2 * cs.y;
            const float b = k1 * cs.y + k2 * cs.x;
            k1 = a;
            k2 = b;
        }
        kp[dst + d] = from_f<T>(k1);
        kp[dst + d + half] = from_f<T>(k2);
        vp[dst + d] = v_new[src + d];
        vp[dst + d + half] = v_new[src + d + half];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        entries[s_entry] = make_entry(page, entry_start(e), slot + 1, true);
    }
}

// One block per (entry slot i of request r): copy the page into dst's page,
// rotating K at the entry's logical positions.
template <typename T>
__global__ void materialize_kernel(PoolView pv, const uint64_t* entries, const int32_t* entry_offsets,
                                   const uint64_t* dst_entries) {
    const int r = blockIdx.y;
    const int idx = entry_offsets[r] + blockIdx.x;
    if (idx >= entry_offsets[r + 1]) return;
    const uint64_t e = entries[idx];
    const uint64_t de = dst_entries[idx];
    const int n = entry_nvalid(e);
    if (n == 0) return;
    if (!entry_ok(pv, e)) return;
    if (entry_page(de) >= (uint32_t)pv.num_pages) {
        record_error(pv.status, LAZYATTN_ERANGE);
        return;
    }
    const uint32_t sp = entry_page(e), dp = entry_page(de);
    const int start = entry_start(e);
    const int D = pv.d, half = D / 2;
    const T* ks = static_cast<const T*>(pv.k_pool);
    const T* vs = static_cast<const T*>(pv.v_pool);
    T* kd = static_cast<T*>(pv.k_pool);
    T* vd = static_cast<T*>(pv.v_pool);
    const int per_head = kPage * half;
    for (int i = threadIdx.x; i < pv.hkv * per_head; i += blockDim.x) {
        const int h = i / per_head;
        const int slot = (i % per_head) / half;
        const int d = i % half;
        const size_t so = (((size_t)sp * pv.hkv + h) * kPage + slot) * D;
        const size_t dso = (((size_t)dp * pv.hkv + h) * kPage + slot) * D;
        if (slot < n) {
            const float2 cs = pv.rope[(size_t)(start + slot) * half + d];
            const float k1 = to_f(ks[so + d]), k2 = to_f(ks[so + d + half]);
            kd[dso + d] = from_f<T>(k1 * cs.x - k2 * cs.y);
            kd[dso + d + half] = from_f<T>(k1 * cs.y + k2 * cs.x);
            vd[dso + d] = vs[so + d];
            vd[dso + d + half] = vs[so + d + half];
        } else {
            kd[dso + d] = from_f<T>(0.f);
            kd[dso + d + half] = from_f<T>(0.f);
            vd[dso + d] = from_f<T>(0.f);
            vd[dso + d + half] = from_f<T>(0.f);
        }
    }
}

// One warp per request: (page, slot, position) of every valid token.
__global__ void resolve_kernel(const uint64_t* entries, const int32_t* entry_offsets, const int32_t* out_off,
                               int32_t* out, int32_t cap, int32_t* status) {
    const int r = blockIdx.x;
    const int lane = threadIdx.x;
    const int e0 = entry_offsets[r], e1 = entry_offsets[r + 1];
    int base = out_off[r];
    for (int c = e0; c < e1; c += 32) {
        const int i = c + lane;
        const uint64_t e = i < e1 ? entries[i] : 0;
        const int n = i < e1 ? entry_nvalid(e) : 0;
        int incl = n;
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const int excl = incl - n;
        for (int s = 0; s < n; ++s) {
            const int row = base + excl + s;
            if (row >= cap) {
                record_error(status, LAZYATTN_ERANGE);
                break;
            }
            out[3 * row + 0] = (int32_t)entry_page(e);
            out[3 * row + 1] = s;
            out[3 * row + 2] = entry_start(e) + s;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
}

inline int cuda_status() { return cudaGetLastError() == cudaSuccess ? LAZYATTN_OK : LAZYATTN_ECUDA; }

}  // namespace

int launch_store_pages(const lazyattn_pool& p, const void* k, const void* v, int32_t n_tokens,
                       const int32_t* pages_host, int32_t npages, cudaStream_t stream) {
    const int esz = p.d.dtype == LAZYATTN_F32 ? 4 : 2;
    const int row_vecs = p.d.head_dim * esz / 16;
    for (int32_t first = 0; first < npages; first += kMaxPagesPerLaunch) {
        const int cnt = std::min<int32_t>(kMaxPagesPerLaunch, npages - first);
        PageList pl;
        for (int i = 0; i < cnt; ++i) pl.ids[i] = pages_host[first + i];
        dim3 grid(cnt, p.d.n_kv_heads);
        if (p.d.key_storage == LAZYATTN_KEYS_DOC_LOCAL)
            store_pages_local_kernel<<<grid, 128, 0, stream>>>(
                static_cast<const __nv_bfloat16*>(k), static_cast<const uint4*>(v),
                static_cast<__nv_bfloat16*>(p.d.k_pool), static_cast<uint4*>(p.d.v_pool),
                static_cast<const float2*>(p.d.rope_table), n_tokens, first, pl, p.d.n_kv_heads, p.d.head_dim,
                p.d.rope_interleaved, p.d.status_word);
        else
            store_pages_kernel<<<grid, 128, 0, stream>>>(static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                                                         static_cast<uint4*>(p.d.k_pool), static_cast<uint4*>(p.d.v_pool),
                                                         n_tokens, first, pl, p.d.n_kv_heads, row_vecs,
                                                         p.d.rope_interleaved, p.d.dtype == LAZYATTN_BF16,
                                                         p.d.status_word);
        if (cuda_status() != LAZYATTN_OK) return LAZYATTN_ECUDA;
    }
    return LAZYATTN_OK;
}

int launch_decode_append(const lazyattn_pool& p, const lazyattn_batch& b, const void* k_new, const void* v_new,
                         int32_t* qpos, cudaStream_t stream) {
    const bool pre = (b.flags & LAZYATTN_KEYS_PREROTATED) != 0;
    const bool local = p.d.key_storage == LAZYATTN_KEYS_DOC_LOCAL;
    const PoolView pv = p.view();
    if (p.d.dtype == LAZYATTN_F32) {
        auto kern = pre ? decode_append_kernel<float, 1> : decode_append_kernel<float, 0>;
        kern<<<b.num_requests, 128, 0, stream>>>(pv, b.entries, b.entry_offsets, static_cast<const float*>(k_new),
                                                 static_cast<const float*>(v_new), qpos, nullptr);
    } else {
        auto kern = local ? decode_append_kernel<__nv_bfloat16, 2>
                          : (pre ? decode_append_kernel<__nv_bfloat16, 1> : decode_append_kernel<__nv_bfloat16, 0>);
        if (launch_dependent(kern, dim3(b.num_requests), dim3(128), 0, stream, pv, b.entries, b.entry_offsets,
                             static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
                             qpos, b.entry_delta) != cudaSuccess)
            return LAZYATTN_ECUDA;
    }
    return cuda_status();
}

int launch_materialize(const lazyattn_pool& p, const lazyattn_batch& b, const uint64_t* dst, cudaStream_t stream) {
    const PoolView pv = p.view();
    dim3 grid(b.max_entries, b.num_requests);
    if (p.d.dtype == LAZYATTN_F32)
        materialize_kernel<float><<<grid, 256, 0, stream>>>(pv, b.entries, b.entry_offsets, dst);
    else
        materialize_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(pv, b.entries, b.entry_offsets, dst);
    return cuda_status();
}

int launch_resolve(const lazyattn_pool& p, const lazyattn_batch& b, const int32_t* out_offsets, int32_t* out,
                   int32_t cap, cudaStream_t stream) {
    resolve_kernel<<<b.num_requests, 32, 0, stream>>>(b.entries, b.entry_offsets, out_offsets, out, cap,
                                                      p.d.status_word);
    return cuda_status();
}

}  // namespace lazyattn
