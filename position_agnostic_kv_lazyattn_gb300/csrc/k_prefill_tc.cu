// bf16 prefill attention on the 5th-generation tensor cores (tcgen05 / TMEM),
// with K/V tiles gathered through the block table by TMA and RoPE applied to
// each K tile in shared memory at the request's logical positions.
//
// LazyAttention §3.2 "Prefilling": the K tile is rotated once, in the inner loop
// over K tiles, by table-driven cos/sin; Q is rotated once. Keys here are stored
// without any position, so every key is rotated at its own logical position
// (start of its page + slot), which Fact 3.2 makes equal to re-encoding.
//
// CTA = (request r, KV head h, query tile): 128 rows = (128 / g) query tokens x
// the g query heads of the group (GQA rows share each K/V tile). Roles:
//   warp 0      TMA producer: 8 pages (K and V, 2 x 64-dim boxes each, 128B
//               swizzle) per 128-key tile into a 2-stage ring
//   warp 1      TMEM owner and single-thread UMMA issuer:
//               S[j%2] = Q K_j^T (fp16 x fp16 -> fp32, 128x128x128),
//               O += P_j V_j (bf16 x bf16 -> fp32, V read MN-major)
//   warps 2-5   softmax: one row per thread (TMEM lane), causal + validity mask
//               on logical positions, online softmax in the log2 domain with
//               lazy rescaling of O (only when the row max grows by > 8), P to
//               shared memory as bf16; final normalisation and store
//   warps 6-9   K rotation: one key row per thread, rotate-half pairs at the
//               key's logical position, written back in place as fp16
// Every wait is bounded; a timeout raises an abort flag that all roles honour,
// drains in-flight copies and MMAs, frees TMEM and records LAZYATTN_EDEVICE.
#include <cudaTypedefs.h>
#include <limits.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace lazyattn {

namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kM = 128;                    // rows per CTA
constexpr int kN = 128;                    // keys per tile
constexpr int kPagesPerTile = kN / kPage;  // 8
constexpr int kThreads = 320;
constexpr int kTileBytes = kN * kD * 2;    // 32 KB per operand tile
constexpr int kChunkBytes = kN * 128;      // 16 KB: one 64-element column chunk of a 128-row tile
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kM * kD * 2;
constexpr int kOffV = kOffK + 2 * kTileBytes;
constexpr int kOffP = kOffV + 2 * kTileBytes;
constexpr int kSmemUsed = kOffP + kM * kN * 2;
constexpr int kSmemBytes = kSmemUsed + 1024;   // + alignment slack
constexpr uint32_t kTmemCols = 512;            // S0 [0,128), S1 [128,256), O [256,384)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;      // log2 units

struct PrefillParams {
    const uint64_t* entries;
    const int32_t* entry_offsets;
    const int32_t* q_offsets;
    const int32_t* q_start;
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    int32_t total_q;
    int32_t g;
    int32_t oob_row;     // a row index outside the K/V tensor maps: TMA fills zeros
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
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
    x[0] = bf_lo(v.x); x[1] = bf_hi(v.x); x[2] = bf_lo(v.y); x[3] = bf_hi(v.y);
    x[4] = bf_lo(v.z); x[5] = bf_hi(v.z); x[6] = bf_lo(v.w); x[7] = bf_hi(v.w);
}

// Entry check shared by every role so that all of them agree on which slots
// hold keys: page in range and positions inside the table.
__device__ __forceinline__ int usable_tokens(const PoolView& pv, uint64_t e) {
    const int n = entry_nvalid(e);
    if (n == 0) return 0;
    if (entry_page(e) >= (uint32_t)pv.num_pages || n > kPage || entry_start(e) + n > pv.max_position) return -1;
    return n;
}

template <bool PREROT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, PoolView pv,
                      PrefillParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    __shared__ uint64_t bar_full[2], bar_empty[2], bar_kready[2], bar_sfull[2], bar_sfree[2];
    __shared__ uint64_t bar_pfull, bar_odone, bar_qready, bar_drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int qt = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = P.g, Hq = pv.hq, Hkv = pv.hkv;
    const int TQ = kM / g;
    const int q0 = P.q_offsets[r], q1 = P.q_offsets[r + 1];
    const int i0 = qt * TQ;
    if (i0 >= q1 - q0) return;                  // uniform: this tile has no rows
    if (q1 > P.total_q) {
        if (threadIdx.x == 0) record_error(pv.status, LAZYATTN_ERANGE);
        return;
    }
    const int ntok = min(TQ, q1 - q0 - i0);
    const int qs = P.q_start[r];
    const int e0 = P.entry_offsets[r], e1 = P.entry_offsets[r + 1];
    const int T = max(e1 - e0, 0) > 0 ? (e1 - e0 + kPagesPerTile - 1) / kPagesPerTile : 0;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
            mbar_init(smem_u32(&bar_kready[s]), 128);
            mbar_init(smem_u32(&bar_sfull[s]), 1);
            mbar_init(smem_u32(&bar_sfree[s]), 128);
        }
        mbar_init(smem_u32(&bar_pfull), 128);
        mbar_init(smem_u32(&bar_odone), 1);
        mbar_init(smem_u32(&bar_qready), 128);
        mbar_init(smem_u32(&bar_drain), 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && T > 0) {
            int last_issued[2] = {-1, -1};
            for (int j = 0; j < T; ++j) {
                const int st = j & 1;
                if (j >= 2 && !mbar_wait(smem_u32(&bar_empty[st]), ((j >> 1) - 1) & 1, abort_flag)) break;
                const uint32_t fb = smem_u32(&bar_full[st]);
                mbar_arrive_expect_tx(fb, 2 * kTileBytes);
                const uint32_t ks = smem_u32(sm + kOffK + st * kTileBytes);
                const uint32_t vs = smem_u32(sm + kOffV + st * kTileBytes);
                for (int p = 0; p < kPagesPerTile; ++p) {
                    const int idx = e0 + j * kPagesPerTile + p;
                    int y = P.oob_row;
                    if (idx < e1) {
                        const uint64_t e = P.entries[idx];
                        if (usable_tokens(pv, e) > 0) y = ((int)entry_page(e) * Hkv + h) * kPage;
                    }
                    tma_load_2d(ks + p * 2048, &kmap, 0, y, fb);
                    tma_load_2d(ks + kChunkBytes + p * 2048, &kmap, 64, y, fb);
                    tma_load_2d(vs + p * 2048, &vmap, 0, y, fb);
                    tma_load_2d(vs + kChunkBytes + p * 2048, &vmap, 64, y, fb);
                }
                last_issued[st] = j;
            }
            if (*abort_flag) {   // let issued copies land before the CTA's smem is released
                volatile int never = 0;
                for (int s = 0; s < 2; ++s)
                    if (last_issued[s] >= 0) mbar_wait(smem_u32(&bar_full[s]), (last_issued[s] >> 1) & 1, &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            const uint32_t idqk = idesc_f16(kM, kN, 0, 0, 0);
            const uint32_t idpv = idesc_f16(kM, kD, 1, 1, 1);
            const uint32_t qa = smem_u32(sm + kOffQ), pa = smem_u32(sm + kOffP);
            bool ok = T > 0 && mbar_wait(smem_u32(&bar_qready), 0, abort_flag);
            for (int j = 0; ok && j <= T; ++j) {
                if (j < T) {
                    const int st = j & 1;
                    ok = mbar_wait(smem_u32(&bar_kready[st]), (j >> 1) & 1, abort_flag);
                    if (ok && j >= 2) ok = mbar_wait(smem_u32(&bar_sfree[st]), ((j >> 1) - 1) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ka = smem_u32(sm + kOffK + st * kTileBytes);
#pragma unroll
                    for (int t = 0; t < kD / 16; ++t) {
                        const uint32_t off = (t >> 2) * kChunkBytes + (t & 3) * 32;
                        umma_f16(tmem + st * kN, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                                 idqk, t > 0);
                    }
                    umma_commit(smem_u32(&bar_sfull[st]));
                }
                if (j >= 1) {
                    const int jp = j - 1, st = jp & 1;
                    ok = mbar_wait(smem_u32(&bar_pfull), jp & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t va = smem_u32(sm + kOffV + st * kTileBytes);
#pragma unroll
                    for (int t = 0; t < kN / 16; ++t) {
                        umma_f16(tmem + 2 * kN, sdesc_sw128(pa + (t >> 2) * kChunkBytes + (t & 3) * 32, 16, 1024),
                                 sdesc_sw128(va + t * 2048, kChunkBytes, 1024), idpv, (jp > 0 || t > 0) ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&bar_odone));
                    umma_commit(smem_u32(&bar_empty[st]));
                }
            }
            // every issued MMA has finished before TMEM / smem are released
            umma_commit(smem_u32(&bar_drain));
            volatile int never = 0;
            mbar_wait(smem_u32(&bar_drain), 0, &never);
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------------ K rotation
        const int kr = threadIdx.x - 192;   // key row of the tile
        for (int j = 0; j < T; ++j) {
            const int st = j & 1;
            if (!mbar_wait(smem_u32(&bar_full[st]), (j >> 1) & 1, abort_flag)) break;
            const int idx = e0 + j * kPagesPerTile + (kr >> 4), slot = kr & 15;
            int pos = -1;
            if (idx < e1) {
                const uint64_t e = P.entries[idx];
                const int n = usable_tokens(pv, e);
                if (n < 0 && slot == 0) record_error(pv.status, LAZYATTN_ERANGE);
                if (slot < n) pos = entry_start(e) + slot;
            }
            uint8_t* kb = sm + kOffK + st * kTileBytes;
            uint8_t* vb = sm + kOffV + st * kTileBytes;
            if (pos >= 0) {
                const float* cs = reinterpret_cast<const float*>(pv.rope + (size_t)pos * (kD / 2));
#pragma unroll 2
                for (int u = 0; u < 8; ++u) {
                    uint4* p1 = reinterpret_cast<uint4*>(kb + sw128_offset(kr, u));
                    uint4* p2 = reinterpret_cast<uint4*>(kb + kChunkBytes + sw128_offset(kr, u));
                    float x1[8], x2[8];
                    unpack8(*p1, x1);
                    unpack8(*p2, x2);
                    if (!PREROT) {
                        const float4* c4 = reinterpret_cast<const float4*>(cs + 16 * u);
                        float t[16];
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const float4 f = __ldg(c4 + v);
                            t[4 * v] = f.x; t[4 * v + 1] = f.y; t[4 * v + 2] = f.z; t[4 * v + 3] = f.w;
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float co = t[2 * e], si = t[2 * e + 1];
                            const float a = x1[e], b = x2[e];
                            x1[e] = a * co - b * si;
                            x2[e] = a * si + b * co;
                        }
                    }
                    *p1 = make_uint4(pack_h2(x1[0], x1[1]), pack_h2(x1[2], x1[3]), pack_h2(x1[4], x1[5]),
                                     pack_h2(x1[6], x1[7]));
                    *p2 = make_uint4(pack_h2(x2[0], x2[1]), pack_h2(x2[2], x2[3]), pack_h2(x2[4], x2[5]),
                                     pack_h2(x2[6], x2[7]));
                }
            } else {   // no key in this slot: zero K (finite scores) and V (no 0 * NaN)
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    *reinterpret_cast<uint4*>(kb + sw128_offset(kr, u)) = z;
                    *reinterpret_cast<uint4*>(kb + kChunkBytes + sw128_offset(kr, u)) = z;
                    *reinterpret_cast<uint4*>(vb + sw128_offset(kr, u)) = z;
                    *reinterpret_cast<uint4*>(vb + kChunkBytes + sw128_offset(kr, u)) = z;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_kready[st]));
        }
    } else {
        // ------------------------------------------------------------ softmax rows
        const int quarter = warp & 3;
        const int row = 32 * quarter + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
        const int t_local = row / g, jh = row - t_local * g;
        const int tok = i0 + t_local;
        const int m_row = qs + tok;
        bool row_valid = t_local < ntok;
        if (row_valid && (m_row < 0 || m_row >= pv.max_position)) {
            record_error(pv.status, LAZYATTN_ERANGE);
            row_valid = false;
        }

        // Q row: rotate at m_row, scale by log2(e)/sqrt(D), fp16, 128B-swizzled K-major
        {
            uint8_t* qsm = sm + kOffQ;
            const float sc = kLog2e * rsqrtf((float)kD);
            const __nv_bfloat16* qp = P.q + ((size_t)(q0 + tok) * Hq + (size_t)h * g + jh) * kD;
            const float* cs = reinterpret_cast<const float*>(pv.rope + (size_t)(row_valid ? m_row : 0) * (kD / 2));
#pragma unroll 2
            for (int u = 0; u < 8; ++u) {
                uint4 w1 = make_uint4(0, 0, 0, 0), w2 = w1;
                if (row_valid) {
                    float x1[8], x2[8];
                    unpack8(__ldg(reinterpret_cast<const uint4*>(qp + 8 * u)), x1);
                    unpack8(__ldg(reinterpret_cast<const uint4*>(qp + 64 + 8 * u)), x2);
                    const float4* c4 = reinterpret_cast<const float4*>(cs + 16 * u);
                    float t[16];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float4 f = __ldg(c4 + v);
                        t[4 * v] = f.x; t[4 * v + 1] = f.y; t[4 * v + 2] = f.z; t[4 * v + 3] = f.w;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float co = t[2 * e], si = t[2 * e + 1];
                        const float a = x1[e], b = x2[e];
                        x1[e] = (a * co - b * si) * sc;
                        x2[e] = (a * si + b * co) * sc;
                    }
                    w1 = make_uint4(pack_h2(x1[0], x1[1]), pack_h2(x1[2], x1[3]), pack_h2(x1[4], x1[5]),
                                    pack_h2(x1[6], x1[7]));
                    w2 = make_uint4(pack_h2(x2[0], x2[1]), pack_h2(x2[2], x2[3]), pack_h2(x2[4], x2[5]),
                                    pack_h2(x2[6], x2[7]));
                }
                *reinterpret_cast<uint4*>(qsm + sw128_offset(row, u)) = w1;
                *reinterpret_cast<uint4*>(qsm + kChunkBytes + sw128_offset(row, u)) = w2;
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_qready));
        }

        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const int st = j & 1;
            // which keys of the tile this row may see
            int kstart[kPagesPerTile], kn[kPagesPerTile];
            bool full = row_valid;
#pragma unroll
            for (int p = 0; p < kPagesPerTile; ++p) {
                const int idx = e0 + j * kPagesPerTile + p;
                int n = 0, s0 = 0;
                if (idx < e1) {
                    const uint64_t e = P.entries[idx];
                    n = max(usable_tokens(pv, e), 0);
                    s0 = entry_start(e);
                }
                kstart[p] = s0;
                kn[p] = n;
                full = full && (n == kPage) && (s0 + kPage - 1 <= m_row);
            }
            ok = mbar_wait(smem_u32(&bar_sfull[st]), (j >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            float s[kN];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld32(trow + st * kN + 32 * c, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(v[i]);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sfree[st]));
            if (!full) {
#pragma unroll
                for (int k = 0; k < kN; ++k) {
                    const int p = k >> 4, sl = k & 15;
                    const bool vis = row_valid && sl < kn[p] && kstart[p] + sl <= m_row;
                    s[k] = vis ? s[k] : -INFINITY;
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < kN; ++k) mx = fmaxf(mx, s[k]);
            float alpha = 1.f;
            if (mx > m_run + kRescaleThreshold) {
                alpha = fast_exp2(m_run - mx);   // 0 when m_run is -inf
                m_run = mx;
            }
            const float mref = (m_run == -INFINITY) ? 0.f : m_run;
            float sum = 0.f;
            uint32_t pk[kN / 2];
#pragma unroll
            for (int k = 0; k < kN; k += 2) {
                const float p0 = fast_exp2(s[k] - mref), p1 = fast_exp2(s[k + 1] - mref);
                sum += p0 + p1;
                pk[k / 2] = pack_bf2(p0, p1);
            }
            l_run = l_run * alpha + sum;
            if (j >= 1) {
                ok = mbar_wait(smem_u32(&bar_odone), (j - 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[32];
                        tmem_ld32(trow + 2 * kN + 32 * c, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        tmem_st32(trow + 2 * kN + 32 * c, v);
                    }
                    tmem_wait_st();
                }
            }
            uint8_t* ps = sm + kOffP;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                *reinterpret_cast<uint4*>(ps + (u >> 3) * kChunkBytes + sw128_offset(row, u & 7)) =
                    make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_pfull));
        }

        // epilogue: O / l -> bf16 rows of out
        if (ok && T > 0) ok = mbar_wait(smem_u32(&bar_odone), (T - 1) & 1, abort_flag);
        tc_fence_after();
        __nv_bfloat16* op = P.out + ((size_t)(q0 + tok) * Hq + (size_t)h * g + jh) * kD;
        const float inv = (ok && l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            if (T > 0 && ok) {
                tmem_ld32(trow + 2 * kN + 32 * c, v);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0u;
            }
            if (t_local < ntok) {
                uint4* dst = reinterpret_cast<uint4*>(op + 32 * c);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float* f = reinterpret_cast<const float*>(v + 8 * i);
                    dst[i] = make_uint4(pack_bf2(f[0] * inv, f[1] * inv), pack_bf2(f[2] * inv, f[3] * inv),
                                        pack_bf2(f[4] * inv, f[5] * inv), pack_bf2(f[6] * inv, f[7] * inv));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && s_abort) record_error(pv.status, LAZYATTN_EDEVICE);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

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

// 2-D view of a pool as rows of 128 bf16: row (page * Hkv + h) * 16 + slot.
bool encode_pool_map(CUtensorMap* map, void* base, uint64_t rows) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kPage};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_prefill_bf16(const lazyattn_pool& p, const lazyattn_batch& b, const __nv_bfloat16* q,
                        __nv_bfloat16* out, cudaStream_t stream) {
    const int g = p.d.n_q_heads / p.d.n_kv_heads;
    if (p.d.head_dim != kD || kM % g != 0) return LAZYATTN_EINVAL;
    const uint64_t rows = (uint64_t)p.d.num_pages * (uint64_t)p.d.n_kv_heads * kPage;
    if (rows + kPage > (uint64_t)INT_MAX) return LAZYATTN_EINVAL;
    if (b.max_q_len < 1) return LAZYATTN_OK;
    CUtensorMap kmap, vmap;
    if (!encode_pool_map(&kmap, p.d.k_pool, rows) || !encode_pool_map(&vmap, p.d.v_pool, rows)) return LAZYATTN_ECUDA;
    PrefillParams P;
    P.entries = b.entries;
    P.entry_offsets = b.entry_offsets;
    P.q_offsets = b.q_offsets;
    P.q_start = b.q_start;
    P.q = q;
    P.out = out;
    P.total_q = b.total_q;
    P.g = g;
    P.oob_row = (int32_t)rows;
    const int TQ = kM / g;
    dim3 grid((b.max_q_len + TQ - 1) / TQ, p.d.n_kv_heads, b.num_requests);
    auto kern = (b.flags & LAZYATTN_KEYS_PREROTATED) ? prefill_tc_kernel<true> : prefill_tc_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
        return LAZYATTN_ECUDA;
    kern<<<grid, kThreads, kSmemBytes, stream>>>(kmap, vmap, p.view(), P);
    return cudaGetLastError() == cudaSuccess ? LAZYATTN_OK : LAZYATTN_ECUDA;
}

}  // namespace lazyattn
