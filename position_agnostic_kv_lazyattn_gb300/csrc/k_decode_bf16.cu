// bf16 decode attention: one query token per request over its paged,
// position-free KV, with RoPE applied to every key in registers at its logical
// position (LazyAttention §3.2 "Decoding"; §3.4: decode stays at ~2LD bytes of
// HBM traffic, the rotation happens on chip).
//
// Work split: a CTA owns (request r, KV head h, split s) and a contiguous run of
// the request's pages; its four warps take pages round-robin. Per page (16
// tokens x 128 dims, one contiguous 4 KB tile each for K and V) a warp:
//   * loads K rows and V rows with 16-byte loads straight into registers,
//   * rotates K at positions start..start+15 (cos/sin from the fp32 position
//     table), converting to fp16 (10-bit mantissa keeps the rotated key close to
//     its fp32 value),
//   * computes S^T = K' Q'^T with m16n8k16 MMAs: 16 tokens x up to 8 query
//     heads of the group, 128-deep,
//   * does the online softmax in the log2 domain (q is pre-scaled by
//     log2(e)/sqrt(D)),
//   * accumulates O^T += V^T P^T with bf16 MMAs (P transposed by movmatrix).
// Warps combine through shared memory; splits combine through a partial buffer
// in the workspace, reduced by the last CTA of each (r, h) to arrive (atomic
// ticket, no waiting).
//
// The head dimension's order inside the MMA is a free permutation as long as the
// K and Q fragments agree; it is chosen so that each lane's 16-byte loads cover
// whole 32-byte sectors and each rotate-half pair (d, d + 64) sits in one lane.
#include "internal.h"

namespace lazyattn {

namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxGroup = 8;

struct DecodeParams {
    const uint64_t* entries;
    const int32_t* entry_offsets;
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    const int32_t* qpos;
    int32_t* tickets;
    float2* ml;
    float* acc;
    int splits;
    int g;
};

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(static_cast<const uint4*>(p)); }
__device__ __forceinline__ float4 ldg16f(const void* p) { return __ldg(static_cast<const float4*>(p)); }
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Lane (gr, c) owns, for its key row, dims {32j + 8c + e : j < 4, e < 8}: four
// 16-byte chunks. Chunks j and j + 2 hold the rotate-half pairs (d, d + 64).
// Rotate one row at logical position pos (unless it is already rotated), scale
// it and emit 16 fp16x2 registers; register 4j + i holds dims (32j + 8c + 2i, +1).
template <bool PREROT>
__device__ __forceinline__ void rotate_row(const uint4 (&kc)[4], const float2* __restrict__ rope, int pos, int c,
                                           float scale, uint32_t (&outr)[16]) {
    float x[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w = u4get(kc[j], i);
            x[j][2 * i] = bf_lo(w);
            x[j][2 * i + 1] = bf_hi(w);
        }
    }
    if (!PREROT) {
        const float2* row = rope + (size_t)pos * (kD / 2);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float* cs = reinterpret_cast<const float*>(row + 32 * j + 8 * c);
            float t[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 f = ldg16f(cs + 4 * v);
                t[4 * v] = f.x;
                t[4 * v + 1] = f.y;
                t[4 * v + 2] = f.z;
                t[4 * v + 3] = f.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float co = t[2 * e], si = t[2 * e + 1];
                const float a = x[j][e], b = x[j + 2][e];
                x[j][e] = a * co - b * si;
                x[j + 2][e] = a * si + b * co;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) outr[4 * j + i] = pack_h2(x[j][2 * i] * scale, x[j][2 * i + 1] * scale);
}

template <bool PREROT>
__global__ void __launch_bounds__(kThreads, 2) decode_bf16_kernel(PoolView pv, DecodeParams P) {
    const int s = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gr = lane >> 2, c = lane & 3;
    const int g = P.g, Hq = pv.hq, Hkv = pv.hkv, S = P.splits;

    __shared__ float sm_acc[kWarps][kMaxGroup][kD];
    __shared__ float sm_m[kWarps][kMaxGroup], sm_l[kWarps][kMaxGroup];
    __shared__ int s_last;

    const int m = P.qpos[r];
    __nv_bfloat16* out_rh = P.out + ((size_t)r * Hq + (size_t)h * g) * kD;
    if (m < 0) {   // request without an appended token (status already recorded)
        if (s == 0)
            for (int i = tid; i < g * kD; i += kThreads) out_rh[i] = __float2bfloat16_rn(0.f);
        return;
    }

    // q of head gr of this group, rotated at m, pre-scaled by log2(e)/sqrt(D), as
    // the B operand (k = head dims, n = head): register 2t / 2t+1 feed k-step t.
    uint32_t qb[16];
    if (gr < g) {
        const __nv_bfloat16* qp = P.q + ((size_t)r * Hq + (size_t)h * g + gr) * kD;
        uint4 qc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) qc[j] = ldg16(qp + 32 * j + 8 * c);
        rotate_row<false>(qc, pv.rope, m, c, 1.4426950408889634f * rsqrtf((float)kD), qb);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) qb[i] = 0u;
    }

    const int e0 = P.entry_offsets[r], e1 = P.entry_offsets[r + 1];
    const int chunk = (e1 - e0 + S - 1) / S;
    const int cb = e0 + s * chunk;
    const int ce = min(e1, cb + chunk);

    const __nv_bfloat16* kpool = static_cast<const __nv_bfloat16*>(pv.k_pool);
    const __nv_bfloat16* vpool = static_cast<const __nv_bfloat16*>(pv.v_pool);

    float o[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
    float mrun0 = -INFINITY, mrun1 = -INFINITY, lrun0 = 0.f, lrun1 = 0.f;

    const int tok[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};

    for (int ei = cb + warp; ei < ce; ei += kWarps) {
        const uint64_t e = P.entries[ei];
        const int nv = entry_nvalid(e);
        if (nv == 0 || !entry_ok(pv, e)) continue;
        const int start = entry_start(e);
        const size_t tile = ((size_t)entry_page(e) * Hkv + h) * kPage * kD;
        const __nv_bfloat16* kt = kpool + tile;
        const __nv_bfloat16* vt = vpool + tile;

        uint4 k0[4], k1[4], vv[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            k0[j] = ldg16(kt + gr * kD + 32 * j + 8 * c);
            k1[j] = ldg16(kt + (gr + 8) * kD + 32 * j + 8 * c);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            vv[t][0] = ldg16(vt + tok[t] * kD + 8 * gr);
            vv[t][1] = ldg16(vt + tok[t] * kD + 64 + 8 * gr);
        }

        // rotate keys at their positions; slots past nv stay in range of the table
        uint32_t ka0[16], ka1[16];
        rotate_row<PREROT>(k0, pv.rope, gr < nv ? start + gr : start, c, 1.f, ka0);
        rotate_row<PREROT>(k1, pv.rope, gr + 8 < nv ? start + gr + 8 : start, c, 1.f, ka1);

        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 8; ++t) mma_f16(sacc, ka0[2 * t], ka1[2 * t], ka0[2 * t + 1], ka1[2 * t + 1], qb[2 * t], qb[2 * t + 1]);

        // S^T fragment: (token gr | gr+8) x (head 2c | 2c+1)
        const bool v0 = gr < nv, v1 = gr + 8 < nv;
        const float s0 = v0 ? sacc[0] : -INFINITY;
        const float s1 = v0 ? sacc[1] : -INFINITY;
        const float s2 = v1 ? sacc[2] : -INFINITY;
        const float s3 = v1 ? sacc[3] : -INFINITY;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(mrun0, mx0), mn1 = fmaxf(mrun1, mx1);
        const float cr0 = fast_exp2(mrun0 - mn0), cr1 = fast_exp2(mrun1 - mn1);
        const float p0 = fast_exp2(s0 - mn0), p1 = fast_exp2(s1 - mn1);
        const float p2 = fast_exp2(s2 - mn0), p3 = fast_exp2(s3 - mn1);
        lrun0 = lrun0 * cr0 + p0 + p2;
        lrun1 = lrun1 * cr1 + p1 + p3;
        mrun0 = mn0;
        mrun1 = mn1;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            o[u][0] *= cr0;
            o[u][1] *= cr1;
            o[u][2] *= cr0;
            o[u][3] *= cr1;
        }
        const uint32_t pb0 = movmatrix_t(pack_bf2(p0, p1));
        const uint32_t pb1 = movmatrix_t(pack_bf2(p2, p3));

        if (nv < kPage) {   // never let stale slots reach the MMA (0 * NaN)
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (tok[t] >= nv) vv[t][0] = vv[t][1] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int qi = u >> 1;
            const uint32_t sel = (u & 1) ? 0x7632u : 0x5410u;
            const uint32_t a0 = prmt(u4get(vv[0][0], qi), u4get(vv[1][0], qi), sel);
            const uint32_t a1 = prmt(u4get(vv[0][1], qi), u4get(vv[1][1], qi), sel);
            const uint32_t a2 = prmt(u4get(vv[2][0], qi), u4get(vv[3][0], qi), sel);
            const uint32_t a3 = prmt(u4get(vv[2][1], qi), u4get(vv[3][1], qi), sel);
            mma_bf16(o[u], a0, a1, a2, a3, pb0, pb1);
        }
    }

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        lrun0 += __shfl_xor_sync(0xffffffffu, lrun0, off);
        lrun1 += __shfl_xor_sync(0xffffffffu, lrun1, off);
    }
    // O^T fragment of m-tile u: dims 8gr+u (c0, c1) and 64+8gr+u (c2, c3); heads 2c, 2c+1
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        sm_acc[warp][2 * c][8 * gr + u] = o[u][0];
        sm_acc[warp][2 * c + 1][8 * gr + u] = o[u][1];
        sm_acc[warp][2 * c][64 + 8 * gr + u] = o[u][2];
        sm_acc[warp][2 * c + 1][64 + 8 * gr + u] = o[u][3];
    }
    if (gr == 0) {
        sm_m[warp][2 * c] = mrun0;
        sm_m[warp][2 * c + 1] = mrun1;
        sm_l[warp][2 * c] = lrun0;
        sm_l[warp][2 * c + 1] = lrun1;
    }
    __syncthreads();

    // combine the four warps: thread -> (head hh, dims d0 .. d0+7)
    const int hh = tid >> 4, d0 = (tid & 15) * 8;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][hh]);
    float L = 0.f, a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float wt = fast_exp2(sm_m[w][hh] - M);
            L += sm_l[w][hh] * wt;
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] += sm_acc[w][hh][d0 + i] * wt;
        }
    }

    if (S == 1) {
        if (hh < g) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
            uint4 w;
            w.x = pack_bf2(a[0] * inv, a[1] * inv);
            w.y = pack_bf2(a[2] * inv, a[3] * inv);
            w.z = pack_bf2(a[4] * inv, a[5] * inv);
            w.w = pack_bf2(a[6] * inv, a[7] * inv);
            *reinterpret_cast<uint4*>(out_rh + (size_t)hh * kD + d0) = w;
        }
        return;
    }

    const size_t rh = (size_t)r * Hkv + h;
    if (hh < g) {
        const size_t slot = (rh * S + s) * g + hh;
        if ((tid & 15) == 0) P.ml[slot] = make_float2(M, L);
        float4* dst = reinterpret_cast<float4*>(P.acc + slot * kD + d0);
        dst[0] = make_float4(a[0], a[1], a[2], a[3]);
        dst[1] = make_float4(a[4], a[5], a[6], a[7]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&P.tickets[rh], 1) == S - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (hh < g) {
        float Mg = -INFINITY;
        for (int t = 0; t < S; ++t) Mg = fmaxf(Mg, __ldcg(&P.ml[(rh * S + t) * g + hh]).x);
        float Lg = 0.f, b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = 0.f;
        if (Mg != -INFINITY) {
            for (int t = 0; t < S; ++t) {
                const size_t slot = (rh * S + t) * g + hh;
                const float2 ml = __ldcg(&P.ml[slot]);
                const float wt = fast_exp2(ml.x - Mg);
                Lg += ml.y * wt;
                const float4* src = reinterpret_cast<const float4*>(P.acc + slot * kD + d0);
                const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
                b[0] += x0.x * wt; b[1] += x0.y * wt; b[2] += x0.z * wt; b[3] += x0.w * wt;
                b[4] += x1.x * wt; b[5] += x1.y * wt; b[6] += x1.z * wt; b[7] += x1.w * wt;
            }
        }
        const float inv = Lg > 0.f ? 1.f / Lg : 0.f;
        uint4 w;
        w.x = pack_bf2(b[0] * inv, b[1] * inv);
        w.y = pack_bf2(b[2] * inv, b[3] * inv);
        w.z = pack_bf2(b[4] * inv, b[5] * inv);
        w.w = pack_bf2(b[6] * inv, b[7] * inv);
        *reinterpret_cast<uint4*>(out_rh + (size_t)hh * kD + d0) = w;
    }
    if (tid == 0) P.tickets[rh] = 0;
}

int choose_splits(const lazyattn_pool& p, const lazyattn_batch& b) {
    const long W = (long)b.num_requests * p.d.n_kv_heads;
    const long slots = std::max(p.decode_slots, 1);
    int best = 1;
    double best_eff = -1.0;
    for (int S = 1; S <= 32; ++S) {
        if (S > 1 && b.max_entries / S < 8) break;   // keep >= 2 pages per warp
        const double waves = (double)(W * S) / (double)slots;
        const double eff = waves / std::ceil(waves);
        if (waves >= 1.0 && eff >= 0.9) return S;
        const double score = waves < 1.0 ? waves : eff;
        if (score > best_eff + 1e-9) {
            best_eff = score;
            best = S;
        }
    }
    return best;
}

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

int decode_occupancy(int* ctas_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, decode_bf16_kernel<false>, kThreads, 0) ==
                   cudaSuccess
               ? LAZYATTN_OK
               : LAZYATTN_ECUDA;
}

DecodeWs decode_ws_layout(const lazyattn_pool& p, const lazyattn_batch& b) {
    DecodeWs L;
    const size_t R = (size_t)b.num_requests, Hkv = (size_t)p.d.n_kv_heads;
    const size_t g = (size_t)(p.d.n_q_heads / p.d.n_kv_heads);
    L.splits = choose_splits(p, b);
    const size_t S = (size_t)L.splits;
    L.qpos_off = 0;
    L.ticket_off = up256(R * sizeof(int32_t));
    L.ml_off = L.ticket_off + up256(R * Hkv * sizeof(int32_t));
    L.acc_off = L.ml_off + up256(R * Hkv * S * g * sizeof(float2));
    L.total = L.acc_off + up256(R * Hkv * S * g * kD * sizeof(float));
    return L;
}

int launch_decode_bf16(const lazyattn_pool& p, const lazyattn_batch& b, const __nv_bfloat16* q,
                       __nv_bfloat16* out, void* ws, const DecodeWs& L, cudaStream_t stream) {
    char* base = static_cast<char*>(ws);
    DecodeParams P;
    P.entries = b.entries;
    P.entry_offsets = b.entry_offsets;
    P.q = q;
    P.out = out;
    P.qpos = reinterpret_cast<const int32_t*>(base + L.qpos_off);
    P.tickets = reinterpret_cast<int32_t*>(base + L.ticket_off);
    P.ml = reinterpret_cast<float2*>(base + L.ml_off);
    P.acc = reinterpret_cast<float*>(base + L.acc_off);
    P.splits = L.splits;
    P.g = p.d.n_q_heads / p.d.n_kv_heads;
    dim3 grid(L.splits, p.d.n_kv_heads, b.num_requests);
    if (b.flags & LAZYATTN_KEYS_PREROTATED)
        decode_bf16_kernel<true><<<grid, kThreads, 0, stream>>>(p.view(), P);
    else
        decode_bf16_kernel<false><<<grid, kThreads, 0, stream>>>(p.view(), P);
    return cudaGetLastError() == cudaSuccess ? LAZYATTN_OK : LAZYATTN_ECUDA;
}

}  // namespace lazyattn
