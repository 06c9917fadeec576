// Document-major bf16 decode on the 5th-generation tensor cores: one CTA per
// (work unit of the decode plan, KV head) reads a run of pages once and serves
// every request of the unit that reads it; a combine kernel then merges each
// request's partial results.
//
// LazyAttention §3 "Problem statement" (several requests of a batch read one
// document at different offsets) and Fact 3.2 (q^T R_{n-m} k depends on the
// positions only through n - m). With keys stored without position, a run's
// keys are rotated once here at run-local positions t (page start relative to
// the run's first page, plus slot), and each reader's q at m - delta (delta =
// that reader's logical position of t = 0): (R_{m-delta} q)^T (R_t k) =
// q^T R_{(delta+t)-m} k, the score the method defines at the key's logical
// position n = delta + t. §3.2 "Decoding" (rotate q, not K, per document) is
// the same move for the paper's own doc-local layout.
//
// CTA = (unit u, KV head h), launched with the KV head fastest, two per SM:
// up to 128 query rows, one per (reader, query head of the group), at TMEM
// lane reader * g + head. Tiles of
// 64 keys (4 pages) stream through two-stage K and V rings. Roles (12 warps):
//   warp 0        TMA producer of K: the unit's entries (read by the whole
//                 warp in one round trip), each page's position-table row for
//                 the run-local rotation, tile info; four consecutive pages
//                 with keys are one 4-page box per half of the dims
//   warp 1        TMEM owner and single-thread UMMA issuer: per tile k,
//                 S_(k%2) = Q K^T (fp16, M 128 x N 64 x K 128), then, once the
//                 softmax of tile k is in, O += P_k V (bf16, P from TMEM);
//                 one commit per QK (K stage free, S ready) and one per PV
//                 (V stage free, O holds the tile)
//   warp 2        TMA producer of V
//   warps 4-7     Q rows (rotated at m - delta, pre-scaled, fp16), softmax of
//                 each tile (thread = TMEM lane = one row; a warp without
//                 reader rows skips the arithmetic), the partial result
//   warps 8-11    K rotation in shared memory at run-local positions (fp16),
//                 zero K of empty slots
// TMEM (256 columns, two CTAs per SM): S_0, S_1 (64 columns each), O (128);
// P_k is written as bf16 over the first 32 columns of its S. V needs no
// fixing up: pages without keys are not read (their rows are outside the
// tensor maps and read as zeros), and slots past a page's valid count are zero
// in every page the library fills, so P = 0 meets V = 0 there.
// Every wait is bounded; a timeout raises an abort flag that all roles honour,
// drains in-flight copies and MMAs, frees TMEM and records LAZYATTN_EDEVICE.
#include <limits.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace lazyattn {

namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kRows = 128;                        // query rows per unit pass
constexpr int kN = 64;                            // keys per K/V tile
constexpr int kPagesPerTile = kN / kPage;         // 4
constexpr int kStages = 2;
constexpr int kInfoSlots = 4;                     // tile-info ring (power of two)
constexpr int kThreads = 384;
constexpr int kQBytes = kRows * kD * 2;           // 32 KB
constexpr int kQChunk = kRows * 128;              // 16 KB (64 dims)
constexpr int kKVBytes = kN * kD * 2;             // 16 KB
constexpr int kKVChunk = kN * 128;                // 8 KB (64 dims)
constexpr int kBaseBytes = kPagesPerTile * 512;   // 4 position-table rows
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kStages * kKVBytes;
constexpr int kOffBase = kOffV + kStages * kKVBytes;
constexpr int kSmemUsed = kOffBase + kStages * kBaseBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;      // + alignment slack
constexpr uint32_t kTmemCols = 256;               // S_0 at 0, S_1 at 64, O at 128
constexpr uint32_t kColO = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;         // log2 units

static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzled tiles need 1 KB alignment");
static_assert(2 * kSmemBytes <= 232448, "two CTAs per SM");

// (written with 16-byte stores, after the tile's copies are issued)
struct __align__(16) TileInfo {
    int j;                       // tile index, -1: no more tiles
    int page0;                   // page of the tile's first entry
    int consec;                  // pages page0 .. page0 + 3, all with keys: one 4-page box per half
    int pad;
    int rel[kPagesPerTile];      // run-local position of slot 0 of each page (doc-local: relative offset)
    int n[kPagesPerTile];        // keys in each page (0: none / unusable)
    int y[kPagesPerTile];        // row of the page in the K/V tensor maps (out of range: zero fill)
};
static_assert(sizeof(TileInfo) == 4 * 16, "tile info layout (written as four 16-byte words)");

struct SharedParams {
    const uint64_t* entries;
    const PlanUnit* units;
    const PlanUser* users;
    const __nv_bfloat16* q;
    const int32_t* qpos;
    float2* ml;                  // [partials][Hkv][g]: (reference maximum, sum), log2 domain
    float* acc;                  // [partials][Hkv][g][D]: unnormalised output rows
    int32_t g;
    int32_t oob_row;             // a row index outside the K/V tensor maps: TMA fills zeros
    const int32_t* entry_delta;  // doc-local pools: document offset of each entry
    int32_t row_blocks;          // rows of the position-table view (max_position / 16); 0: no view
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
__device__ __forceinline__ uint4 pack8_h(const float (&x)[8]) {
    return make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// 32 lanes x 16 columns of 32-bit stored from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// Packed f32x2 arithmetic (two fp32 lanes per instruction).
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
__device__ __forceinline__ float2 f2_neg(float2 a) { return make_float2(-a.x, -a.y); }

__device__ __forceinline__ int usable_tokens(const PoolView& pv, uint64_t e) {
    const int n = entry_nvalid(e);
    if (n == 0) return 0;
    if (entry_page(e) >= (uint32_t)pv.num_pages || n > kPage || entry_start(e) + n > pv.max_position) return -1;
    return n;
}

// PREROT: keys already rotated at their logical positions; q rotated at m.
// LOCAL: keys rotated at document-local positions; each page takes one relative
// rotation by its document offset minus the unit's (the readers' q at m - that).
// INTER: q arrives with interleaved RoPE pairs (de-interleaved on load).
// ALIBI: no rotation; scores get -slope_h (m - n), n = delta + run-local position.
template <bool PREROT, bool LOCAL, bool INTER, bool ALIBI>
__global__ void __launch_bounds__(kThreads, 2)
    decode_shared_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                         const __grid_constant__ CUtensorMap kmap4, const __grid_constant__ CUtensorMap vmap4,
                         const __grid_constant__ CUtensorMap rmap4, PoolView pv, SharedParams P) {
    constexpr bool ROT_K = !PREROT && !ALIBI;   // keys rotated here (run-local or relative doc-local)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    // qkdone[s]: QK of the tile in stage s is done (its K stage is free and
    // its S is ready); pvdone[s]: PV of the tile in stage s is done (its V
    // stage is free, O holds it)
    __shared__ uint64_t bar_kfull[kStages], bar_qkdone[kStages], bar_vfull[kStages], bar_pvdone[kStages];
    __shared__ uint64_t bar_kready[kStages], bar_pfull[kStages], bar_info[kInfoSlots];
    __shared__ uint64_t bar_qready, bar_drain;
    __shared__ TileInfo s_info[kInfoSlots];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = P.g, Hq = pv.hq, Hkv = pv.hkv;
    // CTA = (unit, KV head) with the KV head fastest: the CTAs that run together
    // read whole pages ([page][Hkv][16][D]), and the shortest units of every
    // head come last
    const int h = (int)(blockIdx.x % (unsigned)Hkv);
    const PlanUnit unit = P.units[blockIdx.x / (unsigned)Hkv];   // the plan is not written by the append
    const bool priv = (unit.n_users & kUnitPrivate) != 0;
    const int n_users = unit.n_users & ~kUnitPrivate;
    const int np = unit.n_pages;

    grid_dep_launch_dependents();   // the combine may be scheduled; it waits for this grid
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_kfull[s]), 1);
            mbar_init(smem_u32(&bar_qkdone[s]), 1);
            mbar_init(smem_u32(&bar_vfull[s]), 1);
            mbar_init(smem_u32(&bar_pvdone[s]), 1);
            mbar_init(smem_u32(&bar_kready[s]), 4);   // one arrival per rotation warp
            mbar_init(smem_u32(&bar_pfull[s]), 4);    // one arrival per softmax warp
        }
        for (int s = 0; s < kInfoSlots; ++s) mbar_init(smem_u32(&bar_info[s]), 1);
        mbar_init(smem_u32(&bar_qready), 4);
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
    // waits decided the same way in every lane of a warp (the warp then takes
    // part in warp-wide TMEM loads and stores together)
    auto wwait = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };

    if (warp == 0) {
        // ------------------------------------------------------------ K producer
        // The whole warp reads the unit's entries in one round trip (lane l
        // holds pages l and l + 32; a unit has at most 64); lane 0 waits on
        // barriers and issues the copies. A tail run is read after the append;
        // a shared run's entries and pages are final before it, so its copies
        // start at once. A K stage is reused once QK of the tile two before is
        // done. The info ring needs no wait of its own: slot k % 4 last held
        // tile k - 4, whose readers are all done once QK of tile k - 2 is.
        if (priv) grid_dep_wait();
        const uint64_t* ents = P.entries + unit.entry0;
        uint64_t e[2];
        int dl[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int idx = lane + 32 * c;
            e[c] = idx < np ? ents[idx] : 0ull;
            dl[c] = (LOCAL && idx < np) ? P.entry_delta[unit.entry0 + idx] : 0;
        }
        const int start0 = entry_start(ents[0]);
        const int d0 = LOCAL ? P.entry_delta[unit.entry0] : 0;
        int n[2], rel[2];
        uint32_t pg[2];
        int jl = -1;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int idx = lane + 32 * c;
            pg[c] = entry_page(e[c]);
            n[c] = idx < np ? usable_tokens(pv, e[c]) : 0;
            rel[c] = entry_start(e[c]) - start0;
            if (LOCAL && n[c] > 0) {
                rel[c] = dl[c] - d0;   // the page's relative rotation
                if (rel[c] < 0 || rel[c] >= pv.max_position) n[c] = -1;
            }
            if (ROT_K && n[c] > 0 && (rel[c] < 0 || rel[c] >= pv.max_position)) n[c] = -1;   // table row
            if (n[c] < 0) record_error(pv.status, LAZYATTN_ERANGE);
            if (n[c] > 0) jl = idx / kPagesPerTile;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) jl = max(jl, __shfl_xor_sync(0xffffffffu, jl, off));
        const int j_last = jl;   // the last tile with keys (-1: none; the unit then has no tile)
        int last_k[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) last_k[s] = -1;
        int k = 0;
        bool ok = true;
        for (int j = 0; j <= j_last; ++j) {
            int tn[kPagesPerTile], trel[kPagesPerTile];
            uint32_t tpg[kPagesPerTile];
            bool live = false, consec = true;
#pragma unroll
            for (int p = 0; p < kPagesPerTile; ++p) {
                const int idx = j * kPagesPerTile + p;
                const int src = idx & 31, c = idx >> 5;
                tn[p] = __shfl_sync(0xffffffffu, c ? n[1] : n[0], src);
                trel[p] = __shfl_sync(0xffffffffu, c ? rel[1] : rel[0], src);
                tpg[p] = __shfl_sync(0xffffffffu, c ? pg[1] : pg[0], src);
                if (idx >= np) tn[p] = 0;
                live = live || tn[p] > 0;
                if (tn[p] <= 0 || tpg[p] != tpg[0] + (uint32_t)p) consec = false;
            }
            if (!live) continue;
            const int st = k % kStages;
            if (lane == 0) {
                if (k >= kStages && !mbar_wait(smem_u32(&bar_qkdone[st]), ((k / kStages) - 1) & 1, abort_flag))
                    ok = false;
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            if (lane == 0) {
                TileInfo& info = s_info[k & (kInfoSlots - 1)];
                int ys[kPagesPerTile], nn[kPagesPerTile];
#pragma unroll
                for (int p = 0; p < kPagesPerTile; ++p) {
                    ys[p] = tn[p] > 0 ? ((int)tpg[p] * Hkv + h) * kPage : P.oob_row;
                    nn[p] = max(tn[p], 0);
                }
                // rows of the position table: one box of its 16-row view when the
                // four pages start 16 positions apart, else a copy per page
                bool strided = ROT_K && !LOCAL && P.row_blocks > 0 && trel[0] >= 0 &&
                               trel[0] / kPage + kPagesPerTile <= P.row_blocks;
#pragma unroll
                for (int p = 0; p < kPagesPerTile; ++p) strided = strided && tn[p] > 0 && trel[p] == trel[0] + kPage * p;
                const uint32_t fb = smem_u32(&bar_kfull[st]);
                const uint32_t ds = smem_u32(sm + kOffK + st * kKVBytes);
                const uint32_t bs = smem_u32(sm + kOffBase + st * kBaseBytes);
                // copies first (each copy instruction costs this thread tens of
                // nanoseconds); the stage's own arrival comes after the info
                // writes, so a consumer that sees the stage full sees the info
                mbar_expect_tx(fb, kKVBytes + (ROT_K ? kBaseBytes : 0));
                if (consec) {
                    tma_load_4d(ds, &kmap4, 0, 0, h, (int)tpg[0], fb);
                    tma_load_4d(ds + kKVChunk, &kmap4, 64, 0, h, (int)tpg[0], fb);
                } else {
#pragma unroll
                    for (int p = 0; p < kPagesPerTile; ++p) {
                        tma_load_2d(ds + p * 2048, &kmap, 0, ys[p], fb);
                        tma_load_2d(ds + kKVChunk + p * 2048, &kmap, 64, ys[p], fb);
                    }
                }
                if (strided) {
                    tma_load_3d(bs, &rmap4, 0, trel[0] % kPage, trel[0] / kPage, fb);
                } else if (ROT_K) {
#pragma unroll
                    for (int p = 0; p < kPagesPerTile; ++p) {
                        const float4* base = pv.rope_pair + (tn[p] > 0 ? (size_t)trel[p] * (kD / 4) : 0);
                        bulk_load(bs + p * 512, base, 512, fb);
                    }
                }
                int4* iv = reinterpret_cast<int4*>(&info);
                iv[0] = make_int4(j, (int)tpg[0], consec ? 1 : 0, 0);
                iv[1] = make_int4(trel[0], trel[1], trel[2], trel[3]);
                iv[2] = make_int4(nn[0], nn[1], nn[2], nn[3]);
                iv[3] = make_int4(ys[0], ys[1], ys[2], ys[3]);
                mbar_arrive(smem_u32(&bar_info[k & (kInfoSlots - 1)]));   // releases the info writes
                mbar_arrive(fb);
                last_k[st] = k;
            }
            ++k;
        }
        if (lane == 0) {
            const int st = k % kStages;
            if (ok && (k < kStages ||
                       mbar_wait(smem_u32(&bar_qkdone[st]), ((k / kStages) - 1) & 1, abort_flag))) {
                s_info[k & (kInfoSlots - 1)].j = -1;   // sentinel: no more tiles
                mbar_arrive(smem_u32(&bar_info[k & (kInfoSlots - 1)]));
                mbar_arrive(smem_u32(&bar_kfull[st]));
            } else {
                *abort_flag = 1;
            }
            if (*abort_flag) {   // let issued copies land before the CTA's smem is released
                volatile int never = 0;
                for (int s = 0; s < kStages; ++s)
                    if (last_k[s] >= 0) mbar_wait(smem_u32(&bar_kfull[s]), (last_k[s] / kStages) & 1, &never);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ V producer
        if (lane == 0) {
            if (priv) grid_dep_wait();   // the tail run's V pages take the append's v
            int last_k[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) last_k[s] = -1;
            bool ok = true;
            for (int k = 0;; ++k) {
                const int st = k % kStages;
                ok = mbar_wait(smem_u32(&bar_info[k & (kInfoSlots - 1)]), (k / kInfoSlots) & 1, abort_flag);
                if (!ok) break;
                const TileInfo& info = s_info[k & (kInfoSlots - 1)];
                if (info.j < 0) break;
                int ys[kPagesPerTile];
#pragma unroll
                for (int p = 0; p < kPagesPerTile; ++p) ys[p] = info.y[p];
                const int consec = info.consec, page0 = info.page0;
                if (k >= kStages && !mbar_wait(smem_u32(&bar_pvdone[st]), ((k / kStages) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_vfull[st]);
                const uint32_t ds = smem_u32(sm + kOffV + st * kKVBytes);
                mbar_arrive_expect_tx(fb, kKVBytes);
                if (consec) {
                    tma_load_4d(ds, &vmap4, 0, 0, h, page0, fb);
                    tma_load_4d(ds + kKVChunk, &vmap4, 64, 0, h, page0, fb);
                } else {
#pragma unroll
                    for (int p = 0; p < kPagesPerTile; ++p) {
                        tma_load_2d(ds + p * 2048, &vmap, 0, ys[p], fb);
                        tma_load_2d(ds + kKVChunk + p * 2048, &vmap, 64, ys[p], fb);
                    }
                }
                last_k[st] = k;
            }
            if (!ok) *abort_flag = 1;
            if (*abort_flag) {
                volatile int never = 0;
                for (int s = 0; s < kStages; ++s)
                    if (last_k[s] >= 0) mbar_wait(smem_u32(&bar_vfull[s]), (last_k[s] / kStages) & 1, &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        // QK of tile k + 1 is issued before PV of tile k, so the softmax of tile
        // k + 1 can start while tile k's PV runs. S_(k%2) is next overwritten
        // by QK of tile k + 2, issued after PV of tile k (which reads P_k from
        // it); tcgen05.mma operations of one thread execute in issue order.
        if (lane == 0) {
            const uint32_t idqk = idesc_f16(kRows, kN, 0, 0, 0);
            const uint32_t idpv = idesc_f16(kRows, kD, 1, 1, 1);
            const uint64_t dq0 = sdesc_sw128(smem_u32(sm + kOffQ), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(smem_u32(sm + kOffK), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(sm + kOffV), kKVChunk, 1024);
            auto issue_qk = [&](int k) {
                const int st = k % kStages;
                const uint64_t b0 = dk0 + (uint64_t)(st * (kKVBytes >> 4));
                const uint32_t d = tmem + (uint32_t)(st * kN);
#pragma unroll
                for (int t = 0; t < kD / 16; ++t) {
                    const uint64_t oa = (uint64_t)(((t >> 2) * kQChunk + (t & 3) * 32) >> 4);
                    const uint64_t ob = (uint64_t)(((t >> 2) * kKVChunk + (t & 3) * 32) >> 4);
                    umma_f16(d, dq0 + oa, b0 + ob, idqk, t > 0 ? 1u : 0u);
                }
                umma_commit(smem_u32(&bar_qkdone[st]));   // S ready, K stage free
            };
            // O += P_k V_k: P_k (bf16, 128 rows x 64 keys) is the first 32 columns of S_(k%2).
            auto issue_pv = [&](int k) {
                const int st = k % kStages;
                const uint64_t b0 = dv0 + (uint64_t)(st * (kKVBytes >> 4));
                const uint32_t a = tmem + (uint32_t)(st * kN);
#pragma unroll
                for (int t = 0; t < kN / 16; ++t)
                    umma_f16_ts(tmem + kColO, a + 8 * t, b0 + (uint64_t)(t * 128), idpv, (t > 0 || k > 0) ? 1u : 0u);
                umma_commit(smem_u32(&bar_pvdone[st]));   // O holds the tile, V stage free
            };
            auto kready = [&](int k) {
                return mbar_wait(smem_u32(&bar_kready[k % kStages]), (k / kStages) & 1, abort_flag);
            };
            bool ok = mbar_wait(smem_u32(&bar_qready), 0, abort_flag) && kready(0);
            bool more = ok && s_info[0].j >= 0;
            if (more) {
                tc_fence_after();
                issue_qk(0);
            }
            for (int k = 0; more; ++k) {
                ok = kready(k + 1);
                if (!ok) break;
                const bool next = s_info[(k + 1) & (kInfoSlots - 1)].j >= 0;
                tc_fence_after();
                if (next) issue_qk(k + 1);
                const int st = k % kStages, ph = (k / kStages) & 1;
                ok = mbar_wait(smem_u32(&bar_vfull[st]), ph, abort_flag) &&
                     mbar_wait(smem_u32(&bar_pfull[st]), ph, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(k);
                more = next;
            }
            // every issued MMA has finished before TMEM / smem are released
            umma_commit(smem_u32(&bar_drain));
            volatile int never = 0;
            mbar_wait(smem_u32(&bar_drain), 0, &never);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ K rotation
        // Thread = (slot, group u of 8 frequencies): dims 8u..8u+7 of the first
        // half and 64+8u.. of the second half of every key row with this slot.
        // The angle of slot s of a page is the page's row (cos, sin)(rel theta)
        // composed with (cos, sin)(s theta) (doc-local: the page's row alone).
        const int rt = threadIdx.x - 256;
        const int u = 2 * (rt >> 5) + (lane >> 4), slot = lane & 15;
        float2 cs2[4], sn2[4];   // (cos, sin)(slot * theta_f) for f = 8u + 2v, 8u + 2v + 1
        if (ROT_K && !LOCAL) {
            const float4* t4 = pv.rope_pair + (size_t)slot * (kD / 4) + 4 * u;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 f = slot < pv.max_position ? __ldg(t4 + v) : make_float4(1.f, 1.f, 0.f, 0.f);
                cs2[v] = make_float2(f.x, f.y);
                sn2[v] = make_float2(f.z, f.w);
            }
        }
        // One thread polls the stage's barrier; the named barrier releases the
        // other 127 and makes the go / no-go decision the same for all of them.
        auto rot_wait = [&](uint32_t bar, uint32_t parity) {
            int go = 1;
            if (rt == 0) go = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
            go = go && *abort_flag == 0;
            int all;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\t"
                "selp.b32 %0, 1, 0, q;\n\t}"
                : "=r"(all)
                : "r"(go)
                : "memory");
            return all != 0;
        };
        for (int k = 0;; ++k) {
            const int st = k % kStages, ph = (k / kStages) & 1;
            if (!rot_wait(smem_u32(&bar_kfull[st]), ph)) break;
            const TileInfo& info = s_info[k & (kInfoSlots - 1)];
            if (info.j < 0) {   // no more tiles: let the MMA issuer see the sentinel
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bar_kready[st]));
                break;
            }
            int n[kPagesPerTile];
#pragma unroll
            for (int p = 0; p < kPagesPerTile; ++p) n[p] = info.n[p];
            uint8_t* kb = sm + kOffK + st * kKVBytes;
            const uint8_t* bb = sm + kOffBase + st * kBaseBytes + u * 64;
#pragma unroll 2
            for (int p = 0; p < kPagesPerTile; ++p) {
                const int kr = p * kPage + slot;
                uint4* p1 = reinterpret_cast<uint4*>(kb + sw128_offset(kr, u));
                uint4* p2 = reinterpret_cast<uint4*>(kb + kKVChunk + sw128_offset(kr, u));
                if (slot < n[p]) {
                    float x1[8], x2[8];
                    unpack8(*p1, x1);
                    unpack8(*p2, x2);
                    if (ROT_K) {
                        const float4* b4 = reinterpret_cast<const float4*>(bb + p * 512);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {   // frequencies 8u + 2v, 8u + 2v + 1
                            const float4 bv = b4[v];   // (cos f, cos f+1, sin f, sin f+1)
                            float2 c = make_float2(bv.x, bv.y), s = make_float2(bv.z, bv.w);
                            if (!LOCAL) {   // angle of rel + slot
                                const float2 cc = f2_fma(c, cs2[v], f2_mul(f2_neg(s), sn2[v]));
                                s = f2_fma(s, cs2[v], f2_mul(c, sn2[v]));
                                c = cc;
                            }
                            const float2 a = make_float2(x1[2 * v], x1[2 * v + 1]);
                            const float2 z = make_float2(x2[2 * v], x2[2 * v + 1]);
                            const float2 r1 = f2_fma(a, c, f2_mul(f2_neg(z), s));
                            const float2 r2 = f2_fma(a, s, f2_mul(z, c));
                            x1[2 * v] = r1.x;
                            x1[2 * v + 1] = r1.y;
                            x2[2 * v] = r2.x;
                            x2[2 * v + 1] = r2.y;
                        }
                    }
                    *p1 = pack8_h(x1);
                    *p2 = pack8_h(x2);
                } else {   // no key in this slot: zero K so that its scores stay finite
                    *p1 = make_uint4(0, 0, 0, 0);
                    *p2 = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_kready[st]));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ rows: Q, softmax, partials
        const int quarter = warp - 4;
        const int trow = 32 * quarter + lane;      // TMEM lane = row of the Q tile
        const int j = trow / g, head = trow - j * g;
        const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);
        const bool reader = j < n_users;
        PlanUser us = {0, 0, 0, 0};
        if (reader) us = P.users[unit.user0 + j];
        const __nv_bfloat16* qp_ = P.q + ((size_t)us.request * Hq + (size_t)h * g + head) * kD;
        // The reader's q row (written before this call, not by the append) is
        // fetched into L1 while the append finishes.
        if (reader) {
            asm volatile("prefetch.global.L1 [%0];" ::"l"(qp_));
            asm volatile("prefetch.global.L1 [%0];" ::"l"(qp_ + 64));
        }
        grid_dep_wait();   // the append's positions (and, for the tail run, its keys)
        const int m = reader ? P.qpos[us.request] : -1;
        const int pos_q = PREROT ? m : m - us.delta;   // the row's position relative to the run
        bool row_valid = reader && m >= 0;
        if (row_valid && (pos_q < 0 || pos_q >= pv.max_position)) {
            record_error(pv.status, LAZYATTN_ERANGE);
            row_valid = false;
        }
        // a warp without a row that takes part skips the arithmetic (not the barriers)
        const bool active = __any_sync(0xffffffffu, row_valid);
        if (row_valid) {
            uint8_t* qsm = sm + kOffQ;
            const float sc = kLog2e * pv.qk_scale;
            const float* csq = reinterpret_cast<const float*>(pv.rope + (size_t)pos_q * (kD / 2));
            if (!ALIBI) {   // the row's position-table line (512 B) into L1 beside the q words
#pragma unroll
                for (int l = 0; l < 4; ++l) asm volatile("prefetch.global.L1 [%0];" ::"l"(csq + 32 * l));
            }
            float n2 = 0.f;   // input range: rotated, scaled pairs must stay finite in fp16
#pragma unroll 2
            for (int uu = 0; uu < 8; ++uu) {
                float x1[8], x2[8];
                uint4 a = __ldg(reinterpret_cast<const uint4*>(qp_ + (INTER ? 16 * uu : 8 * uu)));
                uint4 b = __ldg(reinterpret_cast<const uint4*>(qp_ + (INTER ? 16 * uu + 8 : 64 + 8 * uu)));
                if (INTER) deinterleave16(a, b, a, b);
                unpack8(a, x1);
                unpack8(b, x2);
#pragma unroll
                for (int v = 0; v < 8; ++v) n2 = fmaxf(n2, fmaf(x1[v], x1[v], x2[v] * x2[v]));
                const float4* c4 = reinterpret_cast<const float4*>(csq + 16 * uu);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float4 f = ALIBI ? make_float4(1.f, 0.f, 1.f, 0.f) : __ldg(c4 + v);
                    const float a0 = x1[2 * v], z0 = x2[2 * v], a1 = x1[2 * v + 1], z1 = x2[2 * v + 1];
                    x1[2 * v] = (a0 * f.x - z0 * f.y) * sc;
                    x2[2 * v] = (a0 * f.y + z0 * f.x) * sc;
                    x1[2 * v + 1] = (a1 * f.z - z1 * f.w) * sc;
                    x2[2 * v + 1] = (a1 * f.w + z1 * f.z) * sc;
                }
                *reinterpret_cast<uint4*>(qsm + sw128_offset(trow, uu)) = pack8_h(x1);
                *reinterpret_cast<uint4*>(qsm + kQChunk + sw128_offset(trow, uu)) = pack8_h(x2);
            }
            if (!(n2 * sc * sc <= kMaxPairNorm2)) record_error(pv.status, LAZYATTN_ERANGE);
        }
        // Rows past the readers keep whatever the Q buffer held: their scores
        // and outputs are never used (each row of an MMA is independent).
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_qready));
        // ALiBi: slope of this row's query head, in the log2 domain of the scores
        const float alibi_c1 = ALIBI ? alibi_slope(h * g + head, Hq) * kLog2e : 0.f;

        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int k = 0;
        for (;; ++k) {
            const int is = k & (kInfoSlots - 1);
            ok = wwait(smem_u32(&bar_info[is]), (k / kInfoSlots) & 1);
            if (!ok) break;
            const TileInfo& info = s_info[is];
            if (info.j < 0) break;
            // valid keys of the tile: bit i of vis[w] is key 32w + i (pages 2w, 2w+1)
            uint32_t vis[2];
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int l0 = info.n[2 * w], l1 = info.n[2 * w + 1];
                vis[w] = ((1u << l0) - 1u) | (((1u << l1) - 1u) << 16);
            }
            int rel[kPagesPerTile];
#pragma unroll
            for (int p = 0; p < kPagesPerTile; ++p) rel[p] = info.rel[p];
            const bool wfull = (vis[0] & vis[1]) == 0xffffffffu;   // same for every row of the CTA
            const int st = k % kStages;
            ok = wwait(smem_u32(&bar_qkdone[st]), (k / kStages) & 1);
            if (!ok) break;
            tc_fence_after();
            if (active) {
                const uint32_t ts = tl + (uint32_t)(st * kN);
                // ALiBi (log2 domain): key i of page q gets alibi_c1 * (rel_q + i - pos_q)
                auto page_delta = [&](int q) { return rel[q] - pos_q; };
                // two passes over the row's 64 scores, 32 columns at a time (the
                // registers of two CTAs per SM do not hold all 64 at once)
                float mx = -INFINITY;   // the row maximum (ALiBi: an upper bound of the biased scores)
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t v[32];
                    tmem_ld32(ts + 32 * hh, v);
                    if (!wfull) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = (vis[hh] >> i) & 1u ? v[i] : 0xff800000u;
                    }
                    if (ALIBI) {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            float a = -INFINITY;
#pragma unroll
                            for (int i = 0; i < 16; i += 2)
                                a = fmax3(a, __uint_as_float(v[16 * q + i]), __uint_as_float(v[16 * q + i + 1]));
                            mx = fmaxf(mx, a + alibi_c1 * (float)min(page_delta(2 * hh + q) + 15, 0));
                        }
                    } else {
                        float a = -INFINITY, c = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            a = fmax3(a, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                            c = fmax3(c, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                        }
                        mx = fmax3(mx, a, c);
                    }
                }
                float alpha = 1.f;
                if (mx > m_run + kRescaleThreshold) {
                    alpha = fast_exp2(m_run - mx);   // 0 when m_run is -inf
                    m_run = mx;
                }
                const float mref = (m_run == -INFINITY) ? 0.f : m_run;
                // O holds tiles < k once PV of tile k - 1 is done; rescale it when
                // the reference maximum moved for some row of the warp. (S of tile
                // k is done, so PV of tile k - 2, issued before QK of tile k, is
                // done: pvdone[(k-1)%2] is at most one phase behind.)
                if (k >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    ok = wwait(smem_u32(&bar_pvdone[(k - 1) % kStages]), ((k - 1) / kStages) & 1);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tl + kColO + 32 * c, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tl + kColO + 32 * c, o);
                    }
                }
                // P = 2^(s - mref) as bf16 pairs over S's first 32 columns
                float sum = 0.f;
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t v[32];
                    tmem_ld32(ts + 32 * hh, v);
                    if (!wfull) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = (vis[hh] >> i) & 1u ? v[i] : 0xff800000u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float e0 = __uint_as_float(v[2 * i]) - mref, e1 = __uint_as_float(v[2 * i + 1]) - mref;
                        if (ALIBI) {
                            const float b0 = alibi_c1 * (float)(page_delta(2 * hh + (i >> 3)) + 2 * (i & 7));
                            e0 += b0;
                            e1 += b0 + alibi_c1;
                        }
                        const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
                        sum += p0 + p1;
                        pk[i] = pack_bf2(p0, p1);
                    }
                    tmem_st16(ts + 16 * hh, pk);
                }
                l_run = l_run * alpha + sum;
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_pfull[st]));
        }

        // partial result of the row: O (unnormalised), its reference maximum and sum.
        // O is final once every MMA is: the issuer commits the drain barrier
        // (single phase) after the last PV. (Waiting on the last PV's own
        // barrier phase would not do: QK of tile K-1 is issued before PV of
        // tile K-2, so when the last softmax ends only PV of tile K-3 is known
        // to be done, and a parity wait two phases behind returns at once.)
        if (ok && k >= 1) ok = wwait(smem_u32(&bar_drain), 0);
        tc_fence_after();
        const bool have = ok && k >= 1 && row_valid && l_run > 0.f;
        if (reader && m >= 0) {
            const size_t slot = ((size_t)us.partial * Hkv + h) * g + head;
            P.ml[slot] = have ? make_float2(m_run == -INFINITY ? 0.f : m_run, l_run) : make_float2(-INFINITY, 0.f);
        }
        // every lane of the warp takes part in the TMEM loads
        if (__any_sync(0xffffffffu, have)) {
            float4* dst = reinterpret_cast<float4*>(P.acc + (((size_t)us.partial * Hkv + h) * g + head) * kD);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(tl + kColO + 32 * c, o);
                if (have) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[8 * c + i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                                     __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
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

// One CTA per (KV head, request): merge the request's partial results. Thread
// = (part, query head hh of the group, 8 dims): each of the four parts merges
// every fourth partial in one pass (running maximum, its sum and output
// rescaled when it grows), then part 0 merges the four through shared memory.
// Launched as a programmatic dependent of the units' kernel; waits for it
// before reading the partials.
constexpr int kCombineParts = 4;
// (at most 32 registers: four CTAs per SM, so the 152 SMs hold 608 of them in one wave)
__global__ void __launch_bounds__(128 * kCombineParts, 4)
    decode_combine_kernel(PoolView pv, const int32_t* pbase, const int32_t* qpos, const float2* ml, const float* acc,
                          __nv_bfloat16* out, int g) {
    __shared__ float s_m[kCombineParts][128], s_l[kCombineParts][128];
    __shared__ float4 s_a[kCombineParts][2][128];
    grid_dep_launch_dependents();
    grid_dep_wait();
    const int h = blockIdx.x, r = blockIdx.y;
    const int part = threadIdx.x >> 7, t = threadIdx.x & 127;
    const int hh = t >> 4, d0 = (t & 15) * 8;
    const int Hkv = pv.hkv;
    const bool row = hh < g;
    const int k0 = pbase[r], k1 = pbase[r + 1];
    float M = -INFINITY, L = 0.f, a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.f;
    if (row && qpos[r] >= 0) {
#pragma unroll 4
        for (int k = k0 + part; k < k1; k += kCombineParts) {
            const size_t slot = ((size_t)k * Hkv + h) * g + hh;
            const float2 x = __ldcg(&ml[slot]);
            const float4* src = reinterpret_cast<const float4*>(acc + slot * kD + d0);
            const float4 s0 = __ldcg(src), s1 = __ldcg(src + 1);
            if (!(x.y > 0.f)) continue;   // a partial without keys
            if (x.x > M) {                // new reference: earlier terms scaled down (0 from -inf)
                const float sc = fast_exp2(M - x.x);
                L *= sc;
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] *= sc;
                M = x.x;
            }
            const float w = fast_exp2(x.x - M);
            L += x.y * w;
            a[0] += s0.x * w; a[1] += s0.y * w; a[2] += s0.z * w; a[3] += s0.w * w;
            a[4] += s1.x * w; a[5] += s1.y * w; a[6] += s1.z * w; a[7] += s1.w * w;
        }
    }
    s_m[part][t] = M;
    s_l[part][t] = L;
    s_a[part][0][t] = make_float4(a[0], a[1], a[2], a[3]);
    s_a[part][1][t] = make_float4(a[4], a[5], a[6], a[7]);
    __syncthreads();
    if (part != 0 || !row) return;
    float Mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < kCombineParts; ++q) Mx = fmaxf(Mx, s_m[q][t]);
    float Ls = 0.f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
    if (Mx != -INFINITY) {
#pragma unroll
        for (int q = 0; q < kCombineParts; ++q) {
            if (!(s_l[q][t] > 0.f)) continue;
            const float w = fast_exp2(s_m[q][t] - Mx);
            Ls += s_l[q][t] * w;
            const float4 u0 = s_a[q][0][t], u1 = s_a[q][1][t];
            o[0] += u0.x * w; o[1] += u0.y * w; o[2] += u0.z * w; o[3] += u0.w * w;
            o[4] += u1.x * w; o[5] += u1.y * w; o[6] += u1.z * w; o[7] += u1.w * w;
        }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)r * pv.hq + (size_t)h * g + hh) * kD + d0);
    *dst = make_uint4(pack_bf2(o[0] * inv, o[1] * inv), pack_bf2(o[2] * inv, o[3] * inv),
                      pack_bf2(o[4] * inv, o[5] * inv), pack_bf2(o[6] * inv, o[7] * inv));
}

using SharedKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                              const CUtensorMap, PoolView, SharedParams);

SharedKernel shared_kernel_for(bool prerot, bool local, bool inter, bool alibi) {
    if (alibi) return decode_shared_kernel<false, false, false, true>;
    if (local) return inter ? decode_shared_kernel<false, true, true, false> : decode_shared_kernel<false, true, false, false>;
    if (prerot) return inter ? decode_shared_kernel<true, false, true, false> : decode_shared_kernel<true, false, false, false>;
    return inter ? decode_shared_kernel<false, false, true, false> : decode_shared_kernel<false, false, false, false>;
}

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

struct SharedWs {
    size_t ml_off, acc_off, total;
};

SharedWs shared_ws(const lazyattn_pool& p, const lazyattn_plan& plan) {
    const size_t R = (size_t)plan.num_requests, P = (size_t)plan.num_partials;
    const size_t Hkv = (size_t)p.d.n_kv_heads, g = (size_t)(p.d.n_q_heads / p.d.n_kv_heads);
    SharedWs w;
    w.ml_off = up256(R * sizeof(int32_t));
    w.acc_off = w.ml_off + up256(P * Hkv * g * sizeof(float2));
    w.total = w.acc_off + up256(P * Hkv * g * kD * sizeof(float));
    return w;
}

}  // namespace

size_t decode_plan_ws_bytes(const lazyattn_pool& p, const lazyattn_plan& plan) { return shared_ws(p, plan).total; }

int decode_shared_init() {
    for (int i = 0; i < 9; ++i) {
        if (i < 8 && (i & 1) && (i & 2)) continue;   // pre-rotated pages are never doc-local
        SharedKernel k = i == 8 ? shared_kernel_for(false, false, false, true) : shared_kernel_for(i & 1, i & 2, i & 4, false);
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
            return LAZYATTN_ECUDA;
    }
    return LAZYATTN_OK;
}

int launch_decode_shared(const lazyattn_pool& p, const lazyattn_batch& b, const lazyattn_plan& plan,
                         const __nv_bfloat16* q, __nv_bfloat16* out, void* ws, cudaStream_t stream) {
    if (!p.have_maps || !plan.device) return LAZYATTN_ECUDA;
    const SharedWs w = shared_ws(p, plan);
    char* base = static_cast<char*>(ws);
    const char* img = static_cast<const char*>(plan.device);
    SharedParams P;
    P.entries = b.entries;
    P.units = reinterpret_cast<const PlanUnit*>(img + plan.units_off);
    P.users = reinterpret_cast<const PlanUser*>(img + plan.users_off);
    P.q = q;
    P.qpos = reinterpret_cast<const int32_t*>(base);
    P.ml = reinterpret_cast<float2*>(base + w.ml_off);
    P.acc = reinterpret_cast<float*>(base + w.acc_off);
    P.g = p.d.n_q_heads / p.d.n_kv_heads;
    P.oob_row = (int32_t)((uint64_t)p.d.num_pages * (uint64_t)p.d.n_kv_heads * kPage);
    P.entry_delta = b.entry_delta;
    P.row_blocks = p.have_rmap ? p.d.max_position / kPage : 0;
    auto kern = shared_kernel_for((b.flags & LAZYATTN_KEYS_PREROTATED) != 0, p.d.key_storage == LAZYATTN_KEYS_DOC_LOCAL,
                                  p.d.rope_interleaved != 0, p.d.position_encoding == LAZYATTN_POS_ALIBI);
    if (plan.num_units > 0) {
        dim3 grid(plan.num_units * p.d.n_kv_heads);
        if (launch_dependent(kern, grid, dim3(kThreads), kSmemBytes, stream, p.kmap, p.vmap, p.kmap4, p.vmap4, p.rmap4,
                             p.view(), P) != cudaSuccess)
            return LAZYATTN_ECUDA;
    }
    const int32_t* pbase = reinterpret_cast<const int32_t*>(img + plan.pbase_off);
    if (launch_dependent(decode_combine_kernel, dim3(p.d.n_kv_heads, b.num_requests), dim3(128 * kCombineParts), 0, stream, p.view(),
                         pbase, P.qpos, static_cast<const float2*>(P.ml), static_cast<const float*>(P.acc), out,
                         P.g) != cudaSuccess)
        return LAZYATTN_ECUDA;
    return cudaGetLastError() == cudaSuccess ? LAZYATTN_OK : LAZYATTN_ECUDA;
}

}  // namespace lazyattn
