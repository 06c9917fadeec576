// bf16 decode attention: one query token per request over its paged,
// position-free KV, with RoPE applied to every key in registers at its logical
// position (LazyAttention §3.2 "Decoding"; §3.4: decode stays at ~2LD bytes of
// HBM traffic because the rotation happens on chip).
//
// Work split: a CTA owns (request r, KV head h, split s) and a contiguous run of
// the request's pages; its four warps take the run's pages round-robin. Each
// warp keeps its own ring of two page stages in shared memory, filled by TMA
// (lane 0 issues; K and V tiles of one page are 4 KB each, two 64-dim boxes with
// 128-byte swizzle), so the next page is in flight while it computes on the
// current one; three CTAs (12 warps) share an SM. Per page a warp:
//   * reads K as MMA A-fragments with ldmatrix (16 tokens x 128 dims),
//   * rotates every key at position start + slot in registers and rounds it to
//     fp16; the angle's cos/sin come from angle addition: (start) from the
//     page's row of the fp32 position table (one 512 B row per page, fetched
//     one page ahead as one float4 per lane and staged in a per-warp buffer),
//     (slot) from a 9-row copy of the table in shared memory (slots 8..15 add
//     the angle of 8 to that of slots 0..7), so the table adds 1/16 of a page's
//     bytes to the L2 traffic and no global load waits inside the page loop,
//   * computes S^T = K' Q'^T with m16n8k16 MMAs (N = the group's <= 8 heads),
//   * runs the online softmax in the log2 domain (q is pre-scaled by
//     log2(e) times the logit scale, 1/sqrt(D)),
//   * accumulates O^T += V^T P^T (V^T fragments from ldmatrix.trans, P^T from
//     movmatrix).
// Warps combine through shared memory; splits combine through a partial buffer
// in the workspace, reduced by the last CTA of each (r, h) to arrive (atomic
// ticket, nobody waits). Every wait on a TMA is bounded; on a timeout the warp
// drains its copies and the CTA records LAZYATTN_EDEVICE.
#include <limits.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace lazyattn {

namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;                        // the entry prefetch below reads exactly kStages pages ahead
constexpr int kStageBytes = 8192;                 // K tile (2 x 2 KB) + V tile (2 x 2 KB)
constexpr int kRowBytes = 512;                    // one position-table row: 64 (cos, sin)
constexpr int kSlotRows = 9;                      // (cos, sin)(t * theta) for t = 0..8
constexpr int kSlotTableOff = kWarps * kStages * kStageBytes;
constexpr int kBaseBufOff = kSlotTableOff + kSlotRows * kRowBytes;   // per warp: the current page's row
constexpr int kSmemBytes = kBaseBufOff + kWarps * kRowBytes + 1024;
constexpr int kMaxGroup = 8;
constexpr float kLog2e = 1.4426950408889634f;

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
    const int32_t* entry_delta;   // doc-local pools: document offset of each entry
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
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Same predicate in every lane: how many slots of the entry hold keys (0: skip;
// -1: out-of-range page or positions, also skipped and reported).
__device__ __forceinline__ int usable_tokens(const PoolView& pv, uint64_t e) {
    const int n = entry_nvalid(e);
    if (n == 0) return 0;
    if (entry_page(e) >= (uint32_t)pv.num_pages || n > kPage || entry_start(e) + n > pv.max_position) return -1;
    return n;
}

__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t x) { return pack_h2(bf_lo(x), bf_hi(x)); }

// Two fp32 lanes per instruction (packed f32x2 arithmetic).
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\t"
        "mul.rn.f32x2 %0, ra, rb;\n\t}"
        : "=l"(r) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\tmov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\tmov.b64 rc, {%5, %6};\n\t"
        "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
        : "=l"(r) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\t"
        "sub.rn.f32x2 %0, ra, rb;\n\t}"
        : "=l"(r) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
// Angle addition for two frequencies at once: (c, s) of angle 1 + angle 2.
__device__ __forceinline__ void compose2(float2 c1, float2 s1, float2 c2, float2 s2, float2& c, float2& s) {
    c = f2_sub(f2_mul(c1, c2), f2_mul(s1, s2));
    s = f2_fma(s1, c2, f2_mul(c1, s2));
}
// Rotate dims (d, d+1) [bf16x2 x] and their rotate-half partners (d+64, d+65)
// [bf16x2 y] by angles with cosines c and sines s; fp16x2 out.
__device__ __forceinline__ void rotate2v(uint32_t& x, uint32_t& y, float2 c, float2 s) {
    const float2 a = make_float2(bf_lo(x), bf_hi(x)), b = make_float2(bf_lo(y), bf_hi(y));
    const float2 u = f2_sub(f2_mul(a, c), f2_mul(b, s));
    const float2 v = f2_fma(a, s, f2_mul(b, c));
    x = pack_h2(u.x, u.y);
    y = pack_h2(v.x, v.y);
}

// 16-byte unit f4 (frequencies 2*f4, 2*f4+1) of slot-table row t. Odd rows swap
// the two 64-byte halves, so the lanes of a quarter warp (rows 2q and 2q+1,
// four consecutive units each) hit eight different bank groups.
__device__ __forceinline__ int slot_unit(int t, int f4) { return t * (kRowBytes / 16) + (f4 ^ ((t & 1) << 2)); }

// PREROT: keys already rotated at their logical positions. LOCAL: keys rotated
// at document-local positions; instead of the keys, q is rotated at m - delta
// (its position relative to the page's document), once per change of delta
// (§3.2 "Decoding": rotate q per document rather than K per token).
// ALIBI: no rotation of q or k; each score gets -slope_h (m - n) (§3.5).
template <bool PREROT, bool LOCAL, bool ALIBI>
__global__ void __launch_bounds__(kThreads, 3)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       PoolView pv, DecodeParams P) {
    constexpr bool ROT_K = !PREROT && !LOCAL && !ALIBI;   // keys rotated here
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_full[kWarps][kStages];
    __shared__ float sm_m[kWarps][kMaxGroup], sm_l[kWarps][kMaxGroup];
    __shared__ int s_last, s_abort;

    const int s = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gr = lane >> 2, c = lane & 3;
    const int g = P.g, Hq = pv.hq, Hkv = pv.hkv, S = P.splits;

    // Launched as a programmatic dependent of the append kernel: the set-up
    // below touches nothing the append writes; grid_dep_wait() comes before
    // the appended position, the table and the pool are read.
    grid_dep_launch_dependents();
    if (tid == 0) s_abort = 0;
    if (lane == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(smem_u32(&bar_full[warp][st]), 1);
        mbar_fence_init();
    }
    float4* slot_tab = reinterpret_cast<float4*>(sm + kSlotTableOff);   // row t: (cos, sin)(t * theta_i)
    if (ROT_K) {
        for (int i = tid; i < kSlotRows * 32; i += kThreads) {
            const int t = i >> 5, f4 = i & 31;
            const float4 v = t < pv.max_position ? __ldg(reinterpret_cast<const float4*>(pv.rope) + t * 32 + f4)
                                                 : make_float4(1.f, 0.f, 1.f, 0.f);
            slot_tab[slot_unit(t, f4)] = make_float4(v.x, v.z, v.y, v.w);   // (cos, cos, sin, sin)
        }
    }
    __syncthreads();
    const int e0 = P.entry_offsets[r], e1 = P.entry_offsets[r + 1];   // not written by the append
    int m = -1;   // logical position of the appended token: read from the append after grid_dep_wait()

    const int chunk = (e1 - e0 + S - 1) / S;
    const int cb = e0 + s * chunk;
    const int ce = min(e1, cb + chunk);
    const int n_w = ce - cb > warp ? (ce - cb - warp + kWarps - 1) / kWarps : 0;
    const uint64_t* my_entries = P.entries + cb + warp;    // page i of this warp: my_entries[kWarps * i]
    const uint32_t ring = smem_u32(sm + warp * kStages * kStageBytes);
    volatile int* abort_flag = &s_abort;

    // keys of a page that take part (LOCAL: also a valid document offset d)
    auto page_n = [&](uint64_t e, int d) {
        const int n = usable_tokens(pv, e);
        if (LOCAL && n > 0 && (d < 0 || d > entry_start(e) || m - d < 0 || m - d >= pv.max_position)) return -1;
        return n;
    };
    auto issue = [&](int i, uint64_t e, int d) {   // lane 0 only; e, d = entry and offset of page i
        if (i >= n_w) return;
        if (page_n(e, d) <= 0) return;
        const int st = i % kStages;
        const uint32_t bar = smem_u32(&bar_full[warp][st]);
        const int y = ((int)entry_page(e) * Hkv + h) * kPage;
        const uint32_t dst = ring + st * kStageBytes;
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d(dst, &kmap, 0, y, bar);
        tma_load_2d(dst + 2048, &kmap, 64, y, bar);
        tma_load_2d(dst + 4096, &vmap, 0, y, bar);
        tma_load_2d(dst + 6144, &vmap, 64, y, bar);
    };
    // Entries are read two pages ahead and the page's position-table row one
    // page ahead (one float4 per lane, staged in the warp's row buffer when
    // the page comes up), so no global load latency sits inside the page loop.
    auto entry_at = [&](int i) { return i < n_w ? my_entries[kWarps * i] : 0ull; };
    auto delta_at = [&](int i) { return (LOCAL && i < n_w) ? P.entry_delta[cb + warp + kWarps * i] : 0; };
    // the page's row of the position table: its start (ROT_K) or m - delta (LOCAL)
    auto row_of = [&](uint64_t e, int d) {
        const int pos = LOCAL ? m - d : entry_start(e);
        return (!PREROT && !ALIBI && page_n(e, d) > 0)
                   ? __ldg(reinterpret_cast<const float4*>(pv.rope + (size_t)pos * (kD / 2)) + lane)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4* rowbuf = reinterpret_cast<float4*>(sm + kBaseBufOff + warp * kRowBytes);
    // The append writes only the writable entry it appends into and that
    // entry's page; other entries, their pages and the position table are
    // final already. So, where taking part does not depend on m (every layout
    // but doc-local), the first pages of entries that are not writable are
    // requested before waiting for the append, and their loads overlap it.
    uint64_t e_cur = entry_at(0), e_n1 = entry_at(1);
    const bool early0 = !LOCAL && !entry_writable(e_cur);
    const bool early1 = !LOCAL && !entry_writable(e_n1);
    if (lane == 0) {
        if (early0) issue(0, e_cur, 0);
        if (early1) issue(1, e_n1, 0);
    }
    grid_dep_wait();
    m = P.qpos[r];
    __nv_bfloat16* out_rh = P.out + ((size_t)r * Hq + (size_t)h * g) * kD;
    if (m < 0) {   // request without an appended token (status already recorded)
        if (lane == 0) {   // the early copies land before the CTA's shared memory is released
            volatile int never = 0;
            if (early0 && 0 < n_w && page_n(e_cur, 0) > 0) mbar_wait(smem_u32(&bar_full[warp][0]), 0, &never);
            if (early1 && 1 < n_w && page_n(e_n1, 0) > 0) mbar_wait(smem_u32(&bar_full[warp][1]), 0, &never);
        }
        if (s == 0)
            for (int i = tid; i < g * kD; i += kThreads) out_rh[i] = __float2bfloat16_rn(0.f);
        return;
    }
    if (!early0) e_cur = entry_at(0);   // writable entries: read again, the append may have filled them
    if (!early1) e_n1 = entry_at(1);
    int d_cur = delta_at(0), d_n1 = delta_at(1);
    float4 row_next = row_of(e_cur, d_cur);
    if (lane == 0) {
        if (!early0) issue(0, e_cur, d_cur);
        if (!early1) issue(1, e_n1, d_n1);
    }

    // (the first pages are in flight while q is read and rotated)
    // q of head gr, rotated at m and pre-scaled, as the B operand of k-step t:
    // qb[t][0] = dims (16t+2c, +1), qb[t][1] = dims (16t+2c+8, +9).
    uint32_t qb[8][2];
    uint32_t qx[4][2], qy[4][2];   // LOCAL: q as given (bf16 pairs), rotated per document below
    int last_delta = INT_MIN;
    bool q_range_ok = true;        // input range: rotated, scaled pairs must stay finite in fp16
    const float qsc2 = (kLog2e * pv.qk_scale) * (kLog2e * pv.qk_scale);
    auto check_q = [&](uint32_t x, uint32_t y) {
        const float a0 = bf_lo(x), a1 = bf_hi(x), b0 = bf_lo(y), b1 = bf_hi(y);
        const float n2 = fmaxf(fmaf(a0, a0, b0 * b0), fmaf(a1, a1, b1 * b1));
        q_range_ok = q_range_ok && (n2 * qsc2 <= kMaxPairNorm2);
    };
    if (LOCAL) {
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(P.q + ((size_t)r * Hq + (size_t)h * g + min(gr, g - 1)) * kD);
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int d = 16 * t + 2 * c + 8 * hf;
                uint32_t x = gr < g ? __ldg(qp + (pv.interleaved ? d : d / 2)) : 0u;
                uint32_t y = gr < g ? __ldg(qp + (pv.interleaved ? d + 1 : (d + 64) / 2)) : 0u;
                if (pv.interleaved) {   // (2d, 2d+1), (2d+2, 2d+3) -> dims (d, d+1) and (d+64, d+65)
                    const uint32_t p0 = x, p1 = y;
                    x = __byte_perm(p0, p1, 0x5410);
                    y = __byte_perm(p0, p1, 0x7632);
                }
                qx[t][hf] = x;
                qy[t][hf] = y;
                if (gr < g) check_q(x, y);
            }
#pragma unroll
        for (int t = 0; t < 8; ++t) qb[t][0] = qb[t][1] = 0u;
    } else if (gr < g) {
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(P.q + ((size_t)r * Hq + (size_t)h * g + gr) * kD);
        const float4* row = reinterpret_cast<const float4*>(pv.rope + (size_t)m * (kD / 2));
        const float sc = kLog2e * pv.qk_scale;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int d = 16 * t + 2 * c + 8 * hf;
                uint32_t x = __ldg(qp + (pv.interleaved ? d : d / 2)), y = __ldg(qp + (pv.interleaved ? d + 1 : (d + 64) / 2));
                if (pv.interleaved) {   // (2d, 2d+1), (2d+2, 2d+3) -> dims (d, d+1) and (d+64, d+65)
                    const uint32_t p0 = x, p1 = y;
                    x = __byte_perm(p0, p1, 0x5410);
                    y = __byte_perm(p0, p1, 0x7632);
                }
                check_q(x, y);
                const float4 cs = ALIBI ? make_float4(1.f, 0.f, 1.f, 0.f) : __ldg(row + d / 2);
                const float a0 = bf_lo(x), a1 = bf_hi(x), b0 = bf_lo(y), b1 = bf_hi(y);
                qb[t][hf] = pack_h2((a0 * cs.x - b0 * cs.y) * sc, (a1 * cs.z - b1 * cs.w) * sc);
                qb[t + 4][hf] = pack_h2((a0 * cs.y + b0 * cs.x) * sc, (a1 * cs.w + b1 * cs.z) * sc);
            }
        }
    } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) qb[t][0] = qb[t][1] = 0u;
    }

    if (!q_range_ok && s == 0) record_error(pv.status, LAZYATTN_ERANGE);

    // ALiBi slopes of this lane's two heads, in the log2 domain of the scores
    const float al0 = ALIBI ? alibi_slope(h * g + min(2 * c, g - 1), Hq) * kLog2e : 0.f;
    const float al1 = ALIBI ? alibi_slope(h * g + min(2 * c + 1, g - 1), Hq) * kLog2e : 0.f;

    float o[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
    float mrun0 = -INFINITY, mrun1 = -INFINITY, lrun0 = 0.f, lrun1 = 0.f;
    uint32_t phases = 0;
    int consumed_upto = -1;

    for (int i = 0; i < n_w; ++i) {
        const uint64_t e = e_cur;
        const int d = d_cur;
        const uint64_t e_n2 = entry_at(i + 2);
        const int d_n2 = delta_at(i + 2);
        const float4 row_cur = row_next;
        row_next = row_of(e_n1, d_n1);
        const int nv = page_n(e, d);
        const int st = i % kStages;
        if (nv < 0 && lane == 0) record_error(pv.status, LAZYATTN_ERANGE);
        if (nv > 0) {
            if (ROT_K || (LOCAL && d != last_delta)) {
                rowbuf[lane] = make_float4(row_cur.x, row_cur.z, row_cur.y, row_cur.w);   // (cos, cos, sin, sin)
                __syncwarp();
            }
            if (LOCAL && d != last_delta) {   // q rotated at m - d, pre-scaled
                last_delta = d;
                const float sc = kLog2e * pv.qk_scale;
#pragma unroll
                for (int t = 0; t < 4; ++t)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const float4 b4 = rowbuf[8 * t + c + 4 * hf];
                        const float2 a = make_float2(bf_lo(qx[t][hf]), bf_hi(qx[t][hf]));
                        const float2 b = make_float2(bf_lo(qy[t][hf]), bf_hi(qy[t][hf]));
                        const float2 cc = make_float2(b4.x * sc, b4.y * sc), ss = make_float2(b4.z * sc, b4.w * sc);
                        const float2 u = f2_sub(f2_mul(a, cc), f2_mul(b, ss));
                        const float2 v = f2_fma(a, ss, f2_mul(b, cc));
                        qb[t][hf] = pack_h2(u.x, u.y);
                        qb[t + 4][hf] = pack_h2(v.x, v.y);
                    }
            }
            if (!mbar_wait(smem_u32(&bar_full[warp][st]), (phases >> st) & 1u, abort_flag)) break;
            phases ^= 1u << st;
            consumed_upto = i;
            const uint32_t stg = ring + st * kStageBytes;

            // K' = rotated keys as the A operand; k-steps t and t+4 hold the rotate-half
            // partners (dims 16t+.. and 64+16t+..), so they are loaded, rotated and
            // multiplied together: (tokens gr | gr+8) x (dims 16t+2c.. | 16t+2c+8..)
            float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                uint32_t lo[4], hi[4];
                const int row = lane & 15, unit = (t & 3) * 2 + (lane >> 4);
                ldsm_x4(lo, stg + row * 128 + ((unit ^ (row & 7)) << 4));
                ldsm_x4(hi, stg + 2048 + row * 128 + ((unit ^ (row & 7)) << 4));
                if (ROT_K) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        // angle of token gr = angle(start) + angle(gr), and of token gr + 8
                        // = that + angle(8); every factor from a table row
                        const int f4 = 8 * t + c + 4 * hf;
                        // table entries are (cos, cos, sin, sin) of frequencies 2*f4, 2*f4+1
                        const float4 b4 = rowbuf[f4], x = slot_tab[slot_unit(gr, f4)], y = slot_tab[slot_unit(8, f4)];
                        float2 cac, cas, cbc, cbs;
                        compose2(make_float2(b4.x, b4.y), make_float2(b4.z, b4.w), make_float2(x.x, x.y),
                                 make_float2(x.z, x.w), cac, cas);
                        compose2(cac, cas, make_float2(y.x, y.y), make_float2(y.z, y.w), cbc, cbs);
                        rotate2v(lo[2 * hf], hi[2 * hf], cac, cas);
                        rotate2v(lo[2 * hf + 1], hi[2 * hf + 1], cbc, cbs);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        lo[j] = bf2_to_h2(lo[j]);
                        hi[j] = bf2_to_h2(hi[j]);
                    }
                }
                mma_f16(sacc, lo[0], lo[1], lo[2], lo[3], qb[t][0], qb[t][1]);
                mma_f16(sacc, hi[0], hi[1], hi[2], hi[3], qb[t + 4][0], qb[t + 4][1]);
            }

            // S^T fragment: (token gr | gr+8) x (head 2c | 2c+1)
            const bool v0 = gr < nv, v1 = gr + 8 < nv;
            if (ALIBI) {   // tokens start + gr, start + gr + 8; heads 2c, 2c + 1
                const float dn = (float)(entry_start(e) + gr - m);
                sacc[0] += al0 * dn;
                sacc[1] += al1 * dn;
                sacc[2] += al0 * (dn + 8.f);
                sacc[3] += al1 * (dn + 8.f);
            }
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
            if (__any_sync(0xffffffffu, cr0 != 1.f || cr1 != 1.f)) {   // rescale only when a max moved
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    o[u][0] *= cr0;
                    o[u][1] *= cr1;
                    o[u][2] *= cr0;
                    o[u][3] *= cr1;
                }
            }
            const uint32_t pb0 = movmatrix_t(pack_bf2(p0, p1));
            const uint32_t pb1 = movmatrix_t(pack_bf2(p2, p3));

            // V^T as A operand: (dims 16u+gr | 16u+8+gr) x (tokens 2c,2c+1 | 2c+8,2c+9)
            const int vtok = (lane & 7) + ((lane >> 4) << 3);
            if (nv == kPage) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int U = 2 * u + ((lane >> 3) & 1);
                    uint32_t va[4];
                    ldsm_x4_t(va, stg + 4096 + (U >> 3) * 2048 + vtok * 128 + (((U & 7) ^ (vtok & 7)) << 4));
                    mma_bf16(o[u], va[0], va[1], va[2], va[3], pb0, pb1);
                }
            } else {   // slots past nv never reach the MMA (0 * NaN)
                const uint32_t keep0 = ((2 * c < nv) ? 0x0000ffffu : 0u) | ((2 * c + 1 < nv) ? 0xffff0000u : 0u);
                const uint32_t keep1 = ((2 * c + 8 < nv) ? 0x0000ffffu : 0u) | ((2 * c + 9 < nv) ? 0xffff0000u : 0u);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int U = 2 * u + ((lane >> 3) & 1);
                    uint32_t va[4];
                    ldsm_x4_t(va, stg + 4096 + (U >> 3) * 2048 + vtok * 128 + (((U & 7) ^ (vtok & 7)) << 4));
                    mma_bf16(o[u], va[0] & keep0, va[1] & keep0, va[2] & keep1, va[3] & keep1, pb0, pb1);
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async_smem();   // this warp's reads of the stage precede the next TMA into it
            issue(i + kStages, e_n2, d_n2);
        }
        e_cur = e_n1;
        e_n1 = e_n2;
        d_cur = d_n1;
        d_n1 = d_n2;
    }
    if (*abort_flag && lane == 0) {
        // drain copies this warp issued but did not consume before the CTA releases its smem
        volatile int never = 0;
        for (int i = consumed_upto + 1; i < min(n_w, consumed_upto + 1 + kStages); ++i) {
            const uint64_t e = my_entries[kWarps * i];
            if (page_n(e, delta_at(i)) <= 0) continue;
            const int st = i % kStages;
            mbar_wait(smem_u32(&bar_full[warp][st]), (phases >> st) & 1u, &never);
            phases ^= 1u << st;
        }
    }

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        lrun0 += __shfl_xor_sync(0xffffffffu, lrun0, off);
        lrun1 += __shfl_xor_sync(0xffffffffu, lrun1, off);
    }
    __syncthreads();   // every warp is done with its ring: reuse it for the combine
    float* sm_acc = reinterpret_cast<float*>(sm);   // [kWarps][kMaxGroup][kD]
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        float* a0 = sm_acc + ((size_t)warp * kMaxGroup + 2 * c) * kD;
        float* a1 = a0 + kD;
        a0[16 * u + gr] = o[u][0];
        a1[16 * u + gr] = o[u][1];
        a0[16 * u + 8 + gr] = o[u][2];
        a1[16 * u + 8 + gr] = o[u][3];
    }
    if (gr == 0) {
        sm_m[warp][2 * c] = mrun0;
        sm_m[warp][2 * c + 1] = mrun1;
        sm_l[warp][2 * c] = lrun0;
        sm_l[warp][2 * c + 1] = lrun1;
    }
    __syncthreads();
    if (tid == 0 && s_abort) record_error(pv.status, LAZYATTN_EDEVICE);

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
            const float* src = sm_acc + ((size_t)w * kMaxGroup + hh) * kD + d0;
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] += src[i] * wt;
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

// Splits per (request, KV head). Cost model in units of one page per warp:
// every wave of CTAs pays a fixed overhead (prologue, pipeline fill, the
// combine) plus its CTAs' longest page run, so
//   cost(S) = ceil(CTAs / resident slots) * (kCtaOverhead + pages per warp).
// Few long-lived CTAs win for small batches; large batches split until the
// last wave is nearly full.
int choose_splits(const lazyattn_pool& p, const lazyattn_batch& b) {
    constexpr double kCtaOverhead = 4.0;
    const long W = (long)b.num_requests * p.d.n_kv_heads;
    const long slots = std::max(p.decode_slots, 1);
    const long pages = std::max(b.max_entries, 1);
    int best = 1;
    double best_cost = 1e300;
    for (int S = 1; S <= 32; ++S) {
        if (S > 1 && pages / S < 8) break;   // keep >= 2 pages per warp
        const double waves = std::ceil((double)(W * S) / (double)slots);
        const double per_warp = std::ceil((double)pages / (double)(S * kWarps));
        const double cost = waves * (kCtaOverhead + per_warp);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

int decode_occupancy(int* ctas_per_sm) {
    if (cudaFuncSetAttribute(decode_bf16_kernel<false, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(decode_bf16_kernel<true, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(decode_bf16_kernel<false, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(decode_bf16_kernel<false, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
        return LAZYATTN_ECUDA;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, decode_bf16_kernel<false, false, false>, kThreads,
                                                         kSmemBytes) == cudaSuccess
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
    if (!p.have_maps) return LAZYATTN_ECUDA;
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
    P.entry_delta = b.entry_delta;
    auto kern = p.d.position_encoding == LAZYATTN_POS_ALIBI ? decode_bf16_kernel<false, false, true>
                : p.d.key_storage == LAZYATTN_KEYS_DOC_LOCAL
                    ? decode_bf16_kernel<false, true, false>
                    : ((b.flags & LAZYATTN_KEYS_PREROTATED) ? decode_bf16_kernel<true, false, false>
                                                             : decode_bf16_kernel<false, false, false>);
    if (launch_dependent(kern, grid, dim3(kThreads), kSmemBytes, stream, p.kmap, p.vmap, p.view(), P) != cudaSuccess)
        return LAZYATTN_ECUDA;
    return cudaGetLastError() == cudaSuccess ? LAZYATTN_OK : LAZYATTN_ECUDA;
}

}  // namespace lazyattn
