// bf16 prefill attention on the 5th-generation tensor cores (tcgen05 / TMEM),
// with K/V tiles gathered through the block table by TMA and RoPE applied to
// each K tile in shared memory at the request's logical positions.
//
// LazyAttention §3.2 "Prefilling": the K tile is rotated once, in the inner loop
// over K tiles, by table-driven cos/sin; Q is rotated once. Keys here are stored
// without any position, so every key is rotated at its own logical position
// (start of its page + slot), which Fact 3.2 makes equal to re-encoding.
//
// CTA = (request r, KV head h, query pair): two Q tiles of 128 rows, each row a
// (query token, query head of the group) pair, so every K/V tile and its
// rotation serve 256 rows of the group. Tiles of 128 keys (8 pages) stream
// through two-stage K and V rings. Roles (16 warps = 4 warpgroups):
//   warps 0, 2    TMA producers, K ring and V ring: per 64-dim half one box
//                 of eight consecutive pages, else of four, else one per page
//                 (128B swizzle); with K, each page's row (cos, sin)(start *
//                 theta) of the position table (one strided box when the pages
//                 start 16 positions apart, else a bulk copy per page) and the
//                 tile's page starts / token counts in a 4-deep ring. Copy
//                 instructions cost the issuing thread tens of nanoseconds each,
//                 so the K producer computes a tile's boxes and info while it
//                 waits for the stage, issues the copies first and writes the
//                 info after them
//   warp 1        TMEM owner and single-thread UMMA issuer, per tile k:
//                 S_0 = Q_0 K^T; O_1 += P_1 V (tile k-1); S_1 = Q_1 K^T;
//                 O_0 += P_0 V (tile k). QK is fp16 128x128x128 from shared
//                 memory; PV is bf16 128x128x128 with P read from TMEM.
//   warps 4-7     softmax of Q tile 0; warps 8-11 softmax of Q tile 1: one row
//                 per thread (TMEM lane), causal + validity mask on logical
//                 positions, online softmax in the log2 domain with lazy
//                 rescaling of O (only when the row max grows by > 8); P is
//                 written as bf16 over the first 64 columns of its own S
//   warps 12-15   K rotation: thread = (page, 4 frequencies) over the page's
//                 16 keys; the angle of slot 0 is the page's row of the position
//                 table (read once per tile from shared memory), each next
//                 slot's angle the previous one turned by theta (angle addition
//                 in registers); written back in place as fp16
// TMEM: S_0, S_1, O_0, O_1, 128 columns each. P_i aliases S_i: the MMA that
// next overwrites S_i is issued after the PV MMA that reads P_i, and
// tcgen05.mma operations of one thread execute in issue order. The same order
// means that when softmax i sees S_i of tile k, O_i already holds tile k-1.
// Tiles whose keys are all masked for every row of the CTA (past the causal
// edge, or empty entries) are skipped. Only the producer reads the block
// table. Every wait is bounded; a timeout raises an abort flag that all roles
// honour, drains in-flight copies and MMAs, frees TMEM and records
// LAZYATTN_EDEVICE.
#include <limits.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace lazyattn {

namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kTileM = 128;                        // rows per Q tile (one TMEM lane each)
constexpr int kQTiles = 2;
constexpr int kRows = kTileM * kQTiles;
constexpr int kN = 128;                            // keys per K/V tile
constexpr int kPagesPerTile = kN / kPage;          // 8
constexpr int kStages = 2;
constexpr int kInfoSlots = 4;                      // tile-info ring (power of two)
constexpr int kThreads = 512;
constexpr int kQBytes = kTileM * kD * 2;           // 32 KB
constexpr int kQChunk = kTileM * 128;              // 16 KB (64 dims)
constexpr int kKVBytes = kN * kD * 2;              // 32 KB
constexpr int kKVChunk = kN * 128;                 // 16 KB (64 dims)
constexpr int kBaseBytes = kPagesPerTile * 512;    // 8 position-table rows
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQTiles * kQBytes;
constexpr int kOffV = kOffK + kStages * kKVBytes;
constexpr int kOffBase = kOffV + kStages * kKVBytes;
constexpr int kSmemUsed = kOffBase + kStages * kBaseBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;       // + alignment slack
constexpr uint32_t kTmemCols = 512;                // S_i at i*128 (P_i in its first 64), O_i at 256 + i*128
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;          // log2 units

static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzled tiles need 1 KB alignment");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// What the producer tells the consumers about a tile (written with 16-byte
// stores: the producer's stores queue behind the math roles' shared-memory
// traffic).
struct __align__(16) TileInfo {
    int j;                        // tile index, -1: no more tiles
    int consec;                   // bit b < 2: pages 4b .. 4b+3 are consecutive pages, all with keys;
                                  // bit 2: all eight are
    int page[2];                  // first page of each group of four
    int start[kPagesPerTile];     // logical position of slot 0 of each page
    int n[kPagesPerTile];         // keys in each page (0: none / unusable)
    int y[kPagesPerTile];         // row of the page in the K/V tensor maps (out of range: zero fill)
    int full_from;                // every page full: rows at positions >= this see every key; else INT_MAX
    int pad[3];
};

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
    const int32_t* entry_delta;   // doc-local pools: document offset of each entry
    int32_t row_blocks;           // rows of the position-table view (max_position / 16); 0: no view
    int32_t splits;               // CTAs per (request, KV head, query pair), each a share of the tiles
    int32_t qpairs;               // query pairs per request (grid.x / splits)
    float* part_o;                // splits > 1: [item][split][row][D] unnormalised O
    float2* part_ml;              // splits > 1: [item][split][row] (reference maximum, sum)
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

// max of three (one instruction on this architecture)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Two fp32 lanes per instruction (packed f32x2 arithmetic).
__device__ __forceinline__ float2 sub2(float2 a, float m) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %3};\n\t"
        "sub.rn.f32x2 %0, ra, rb;\n\t}"
        : "=l"(r) : "f"(a.x), "f"(a.y), "f"(m));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\t"
        "add.rn.f32x2 %0, ra, rb;\n\t}"
        : "=l"(r) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\t"
        "mul.rn.f32x2 %0, ra, rb;\n\t}"
        : "=l"(r) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
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
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\tmov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\tmov.b64 rc, {%5, %6};\n\t"
        "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
        : "=l"(r) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
// Entry check shared by every role so that all of them agree on which slots
// hold keys: page in range and positions inside the table.
__device__ __forceinline__ int usable_tokens(const PoolView& pv, uint64_t e) {
    const int n = entry_nvalid(e);
    if (n == 0) return 0;
    if (entry_page(e) >= (uint32_t)pv.num_pages || n > kPage || entry_start(e) + n > pv.max_position) return -1;
    return n;
}

// PREROT: keys already rotated at their logical positions (no rotation).
// LOCAL: keys rotated at document-local positions; each page takes one relative
// rotation by its document's offset (§3.2 "Prefilling": R_delta R_t = R_(delta+t)).
// INTER: q arrives with interleaved RoPE pairs and is de-interleaved on load.
// ALIBI: no rotation of q or k; each score gets the bias -slope_h (m - n)
// (§3.5, score-space positional methods), computed from logical positions.
// SPLIT: the request's tiles are shared by P.splits CTAs, each writing partials
// (a separate instantiation, so that the unsplit kernel's code is unchanged).
template <bool PREROT, bool LOCAL, bool INTER, bool ALIBI, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap kmap4, const __grid_constant__ CUtensorMap vmap4,
                      const __grid_constant__ CUtensorMap kmap8, const __grid_constant__ CUtensorMap vmap8,
                      const __grid_constant__ CUtensorMap rmap, PoolView pv, PrefillParams P) {
    constexpr bool ROT = !PREROT && !ALIBI;   // K rotated here: the pages' position-table rows are loaded
    static_assert(sizeof(TileInfo) == 8 * 16, "tile info layout (written as eight 16-byte words)");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    __shared__ uint64_t bar_kfull[kStages], bar_kempty[kStages], bar_vfull[kStages], bar_vempty[kStages];
    __shared__ uint64_t bar_kready[kStages], bar_info[kInfoSlots];
    __shared__ uint64_t bar_sfull[kQTiles], bar_pfull[kQTiles], bar_odone[kQTiles];
    __shared__ uint64_t bar_qready, bar_drain;
    __shared__ TileInfo s_info[kInfoSlots];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int qp = SPLIT ? (int)blockIdx.x / P.splits : (int)blockIdx.x;
    const int split = SPLIT ? (int)blockIdx.x - qp * P.splits : 0;
    const int h = blockIdx.y, r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = P.g, Hq = pv.hq, Hkv = pv.hkv;
    const int TQ = kRows / g;                  // query tokens per CTA
    const int q0 = P.q_offsets[r], q1 = P.q_offsets[r + 1];
    const int i0 = qp * TQ;
    if (i0 >= q1 - q0) return;                 // uniform: this CTA has no rows
    if (q1 > P.total_q) {
        if (threadIdx.x == 0) record_error(pv.status, LAZYATTN_ERANGE);
        return;
    }
    const int ntok = min(TQ, q1 - q0 - i0);
    const int nrows = ntok * g;
    const bool tile1 = nrows > kTileM;         // second Q tile has rows
    const int qs = P.q_start[r];
    const int m_hi = qs + i0 + ntok - 1;       // largest query position of the CTA
    const int e0 = P.entry_offsets[r], e1 = P.entry_offsets[r + 1];
    // This CTA's share of the request's tiles: [jb, jb + T)
    const int t_all = e1 > e0 ? (e1 - e0 + kPagesPerTile - 1) / kPagesPerTile : 0;
    const int chunk = SPLIT ? (t_all + P.splits - 1) / P.splits : t_all;
    const int jb = SPLIT ? min(t_all, split * chunk) : 0;
    const int T = SPLIT ? min(t_all, jb + chunk) - jb : t_all;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_kfull[s]), 1);
            mbar_init(smem_u32(&bar_kempty[s]), 1);
            mbar_init(smem_u32(&bar_vfull[s]), 1);
            mbar_init(smem_u32(&bar_vempty[s]), 1);
            mbar_init(smem_u32(&bar_kready[s]), 4);   // one arrival per rotation warp
        }
        for (int s = 0; s < kInfoSlots; ++s) mbar_init(smem_u32(&bar_info[s]), 1);
        for (int i = 0; i < kQTiles; ++i) {
            mbar_init(smem_u32(&bar_sfull[i]), 1);
            mbar_init(smem_u32(&bar_pfull[i]), 4);   // one arrival per softmax warp
            mbar_init(smem_u32(&bar_odone[i]), 1);
        }
        mbar_init(smem_u32(&bar_qready), kQTiles * 4);
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
        // ------------------------------------------------------------ K producer
        // Reads the block table (entries of tile j + 1 are loaded while tile j is
        // issued), decides which tiles are live, publishes each live tile's info
        // (page starts, token counts, tensor-map rows) in a 4-deep ring, and
        // streams K tiles with their pages' position-table rows. A K stage is
        // reused once the tile's QK MMAs are done. The info ring needs no wait
        // of its own: slot k % 4 last held tile k - 4, and the K stage wait for
        // tile k (QK of tile k - 2 done) already implies that the PV MMAs of
        // tile k - 3, and so every reader of tile k - 4's info, are done.
        // A tile is live iff one of its pages holds a key at a position <= the
        // largest query position of the CTA.
        if (lane == 0 && T > 0) {
            auto load_entries = [&](int jj, uint64_t (&e)[kPagesPerTile], int (&dl)[kPagesPerTile]) {
#pragma unroll
                for (int p = 0; p < kPagesPerTile; ++p) {
                    const int idx = e0 + (jb + jj) * kPagesPerTile + p;
                    const uint64_t v = P.entries[min(idx, e1 - 1)];
                    e[p] = idx < e1 ? v : 0ull;   // 0: an empty entry
                    if (LOCAL) dl[p] = P.entry_delta[min(idx, e1 - 1)];
                }
            };
            int last_k[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) last_k[s] = -1;
            uint64_t cur[kPagesPerTile], nxt[kPagesPerTile] = {};
            int curd[kPagesPerTile] = {}, nxtd[kPagesPerTile] = {};   // LOCAL: document offsets
            load_entries(0, cur, curd);
            int k = 0;
            bool ok = true;
            for (int j = 0; j <= T; ++j) {
                if (j + 1 < T) load_entries(j + 1, nxt, nxtd);
                int n[kPagesPerTile];
                bool live = false;
#pragma unroll
                for (int p = 0; p < kPagesPerTile; ++p) {
                    n[p] = j < T ? usable_tokens(pv, cur[p]) : 0;
                    if (LOCAL && n[p] > 0 &&
                        (curd[p] < 0 || curd[p] > entry_start(cur[p]) || curd[p] >= pv.max_position))
                        n[p] = -1;
                    live = live || (n[p] > 0 && entry_start(cur[p]) <= m_hi);
                }
                if (j == T || live) {
                    const int st = k % kStages;
                    // Everything the tile's copies and info need, before the wait.
                    int ys[kPagesPerTile], nn[kPagesPerTile], ss[kPagesPerTile];
                    int consec = 3;
                    bool bad = false;
#pragma unroll
                    for (int p = 0; p < kPagesPerTile; ++p) {
                        bad = bad || n[p] < 0;
                        nn[p] = max(n[p], 0);
                        ss[p] = entry_start(cur[p]);
                        ys[p] = n[p] > 0 ? ((int)entry_page(cur[p]) * Hkv + h) * kPage : P.oob_row;
                        if (n[p] <= 0 || entry_page(cur[p]) != entry_page(cur[p & ~3]) + (uint32_t)(p & 3))
                            consec &= ~(1 << (p >> 2));
                    }
                    const int pg0 = (int)entry_page(cur[0]), pg1 = (int)entry_page(cur[4]);
                    if (consec == 3 && pg1 == pg0 + 4) consec |= 4;
                    // The pages' rows: when the eight pages start 16 positions apart
                    // (full pages at consecutive positions), one box of the position
                    // table's 16-row view; else a copy per page.
                    const int t0 = ss[0];
                    bool strided = ROT && !LOCAL && P.row_blocks > 0 && t0 / kPage + kPagesPerTile <= P.row_blocks;
#pragma unroll
                    for (int p = 0; p < kPagesPerTile; ++p) strided = strided && n[p] > 0 && ss[p] == t0 + kPage * p;
                    if (k >= kStages && !mbar_wait(smem_u32(&bar_kempty[st]), ((k / kStages) - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&bar_kfull[st]);
                    TileInfo& info = s_info[k & (kInfoSlots - 1)];
                    const uint32_t ib = smem_u32(&bar_info[k & (kInfoSlots - 1)]);
                    if (j == T) {   // sentinel: no more tiles
                        info.j = -1;
                        mbar_arrive(ib);
                        mbar_arrive(fb);
                        break;
                    }
                    const uint32_t ds = smem_u32(sm + kOffK + st * kKVBytes);
                    const uint32_t bs = smem_u32(sm + kOffBase + st * kBaseBytes);
                    // Copies first (each copy instruction costs this thread tens of
                    // nanoseconds, so eight consecutive pages take one box per half
                    // of the dims); the stage's own arrival comes after the info
                    // writes, so a consumer that sees the stage full sees the info.
                    mbar_expect_tx(fb, kKVBytes + (ROT ? kBaseBytes : 0));
                    if (consec & 4) {
                        tma_load_4d(ds, &kmap8, 0, 0, h, pg0, fb);
                        tma_load_4d(ds + kKVChunk, &kmap8, 64, 0, h, pg0, fb);
                    } else {
#pragma unroll
                        for (int b4 = 0; b4 < 2; ++b4) {
                            if (consec & (1 << b4)) {   // four consecutive pages: one box per half of the dims
                                const int pg = b4 ? pg1 : pg0;
                                tma_load_4d(ds + b4 * 8192, &kmap4, 0, 0, h, pg, fb);
                                tma_load_4d(ds + kKVChunk + b4 * 8192, &kmap4, 64, 0, h, pg, fb);
                            } else {
#pragma unroll
                                for (int p = 4 * b4; p < 4 * b4 + 4; ++p) {
                                    tma_load_2d(ds + p * 2048, &kmap, 0, ys[p], fb);
                                    tma_load_2d(ds + kKVChunk + p * 2048, &kmap, 64, ys[p], fb);
                                }
                            }
                        }
                    }
                    if (strided) {
                        tma_load_3d(bs, &rmap, 0, t0 % kPage, t0 / kPage, fb);
                    } else if (ROT) {
#pragma unroll
                        for (int p = 0; p < kPagesPerTile; ++p) {
                            const int rowpos = LOCAL ? curd[p] : ss[p];   // position of the page's rotation
                            const float4* base = pv.rope_pair + (n[p] > 0 ? (size_t)rowpos * (kD / 4) : 0);
                            bulk_load(bs + p * 512, base, 512, fb);
                        }
                    }
                    int4* iv = reinterpret_cast<int4*>(&info);
                    iv[0] = make_int4(j, consec, pg0, pg1);
                    iv[1] = make_int4(ss[0], ss[1], ss[2], ss[3]);
                    iv[2] = make_int4(ss[4], ss[5], ss[6], ss[7]);
                    iv[3] = make_int4(nn[0], nn[1], nn[2], nn[3]);
                    iv[4] = make_int4(nn[4], nn[5], nn[6], nn[7]);
                    iv[5] = make_int4(ys[0], ys[1], ys[2], ys[3]);
                    iv[6] = make_int4(ys[4], ys[5], ys[6], ys[7]);
                    int full_from = 0;
#pragma unroll
                    for (int p = 0; p < kPagesPerTile; ++p)
                        full_from = nn[p] == kPage ? max(full_from, ss[p] + kPage - 1) : INT_MAX;
                    iv[7] = make_int4(full_from, 0, 0, 0);
                    mbar_arrive(ib);   // releases the info writes to the other roles
                    mbar_arrive(fb);
                    if (bad) record_error(pv.status, LAZYATTN_ERANGE);
                    last_k[st] = k;
                    ++k;
                }
#pragma unroll
                for (int p = 0; p < kPagesPerTile; ++p) {
                    cur[p] = nxt[p];
                    curd[p] = nxtd[p];
                }
            }
            if (!ok) *abort_flag = 1;
            if (*abort_flag) {   // let issued copies land before the CTA's smem is released
                volatile int never = 0;
                for (int s = 0; s < kStages; ++s)
                    if (last_k[s] >= 0) mbar_wait(smem_u32(&bar_kfull[s]), (last_k[s] / kStages) & 1, &never);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ V producer
        // Takes the page rows from the tile info; a V stage is reused once the
        // tile's PV MMAs are done.
        if (lane == 0 && T > 0) {
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
                const int consec = info.consec, pg0 = info.page[0], pg1 = info.page[1];
                if (k >= kStages && !mbar_wait(smem_u32(&bar_vempty[st]), ((k / kStages) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_vfull[st]);
                const uint32_t ds = smem_u32(sm + kOffV + st * kKVBytes);
                mbar_arrive_expect_tx(fb, kKVBytes);
                if (consec & 4) {
                    tma_load_4d(ds, &vmap8, 0, 0, h, pg0, fb);
                    tma_load_4d(ds + kKVChunk, &vmap8, 64, 0, h, pg0, fb);
                } else {
#pragma unroll
                    for (int b4 = 0; b4 < 2; ++b4) {
                        if (consec & (1 << b4)) {
                            const int pg = b4 ? pg1 : pg0;
                            tma_load_4d(ds + b4 * 8192, &vmap4, 0, 0, h, pg, fb);
                            tma_load_4d(ds + kKVChunk + b4 * 8192, &vmap4, 64, 0, h, pg, fb);
                        } else {
#pragma unroll
                            for (int p = 4 * b4; p < 4 * b4 + 4; ++p) {
                                tma_load_2d(ds + p * 2048, &vmap, 0, ys[p], fb);
                                tma_load_2d(ds + kKVChunk + p * 2048, &vmap, 64, ys[p], fb);
                            }
                        }
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
        if (lane == 0) {
            const uint32_t idqk = idesc_f16(kTileM, kN, 0, 0, 0);
            const uint32_t idpv = idesc_f16(kTileM, kD, 1, 1, 1);
            const int nt = tile1 ? 2 : 1;
            // Descriptors are built once; a k-step only moves the start address,
            // i.e. adds (byte offset >> 4) to the low field of the descriptor.
            // Q tiles and ring stages are evenly spaced: index * stride.
            const uint64_t dq0 = sdesc_sw128(smem_u32(sm + kOffQ), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(smem_u32(sm + kOffK), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(sm + kOffV), kKVChunk, 1024);
            auto issue_qk = [&](int i, int st) {
                const uint64_t a0 = dq0 + (uint64_t)(i * (kQBytes >> 4)), b0 = dk0 + (uint64_t)(st * (kKVBytes >> 4));
                const uint32_t d = tmem + i * 128;
#pragma unroll
                for (int t = 0; t < kD / 16; ++t) {
                    const uint64_t oa = (uint64_t)(((t >> 2) * kQChunk + (t & 3) * 32) >> 4);
                    const uint64_t ob = (uint64_t)(((t >> 2) * kKVChunk + (t & 3) * 32) >> 4);
                    umma_f16(d, a0 + oa, b0 + ob, idqk, t > 0 ? 1u : 0u);
                }
                umma_commit(smem_u32(&bar_sfull[i]));
            };
            // O_i += P_i V: P_i (bf16, 128 x 128 keys) is the first 64 columns of S_i.
            auto issue_pv = [&](int i, int st, bool first) {
                const uint64_t b0 = dv0 + (uint64_t)(st * (kKVBytes >> 4));
                const uint32_t d = tmem + 256 + i * 128, a = tmem + i * 128;
#pragma unroll
                for (int t = 0; t < kN / 16; ++t)
                    umma_f16_ts(d, a + 8 * t, b0 + (uint64_t)(t * 128), idpv, (t > 0 || !first) ? 1u : 0u);
                umma_commit(smem_u32(&bar_odone[i]));
            };
            bool ok = T > 0 && mbar_wait(smem_u32(&bar_qready), 0, abort_flag);
            int k = 0;
            for (; ok;) {
                const int st = k % kStages, ph = (k / kStages) & 1;
                // K rotated (the rotation warps arrive for the sentinel too)
                ok = mbar_wait(smem_u32(&bar_kready[st]), ph, abort_flag);
                if (!ok || s_info[k & (kInfoSlots - 1)].j < 0) break;
                tc_fence_after();
                issue_qk(0, st);
                if (nt == 2) {
                    if (k >= 1) {   // P_1 V of the previous tile, then S_1 may be overwritten
                        ok = mbar_wait(smem_u32(&bar_pfull[1]), (k - 1) & 1, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        const int pst = (k - 1) % kStages;
                        issue_pv(1, pst, k == 1);
                        umma_commit(smem_u32(&bar_vempty[pst]));
                    }
                    issue_qk(1, st);
                }
                umma_commit(smem_u32(&bar_kempty[st]));   // K stage free once these QK MMAs finish
                ok = mbar_wait(smem_u32(&bar_vfull[st]), ph, abort_flag) &&
                     mbar_wait(smem_u32(&bar_pfull[0]), k & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(0, st, k == 0);
                if (nt == 1) umma_commit(smem_u32(&bar_vempty[st]));
                ++k;
            }
            if (ok && nt == 2 && k >= 1) {   // P_1 V of the last tile
                ok = mbar_wait(smem_u32(&bar_pfull[1]), (k - 1) & 1, abort_flag);
                if (ok) {
                    tc_fence_after();
                    const int pst = (k - 1) % kStages;
                    issue_pv(1, pst, k == 1);
                    umma_commit(smem_u32(&bar_vempty[pst]));
                }
            }
            // every issued MMA has finished before TMEM / smem are released
            umma_commit(smem_u32(&bar_drain));
            volatile int never = 0;
            mbar_wait(smem_u32(&bar_drain), 0, &never);
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ K rotation
        // Thread = (page p, group u of 4 frequencies): dims 4u..4u+3 of both
        // halves of the page's 16 key rows. The angle of slot 0 is the page's
        // row of the (paired) position table; each next slot's angle is the
        // previous one turned by theta (angle addition in registers), so a
        // thread reads its page's row once per tile.
        const int rt = threadIdx.x - 384;
        const int p = rt >> 4, u = rt & 15;
        // (cos, sin, -sin)(theta_f) for f = 4u, 4u+1 and 4u+2, 4u+3, as lane pairs
        float2 c1[2], s1[2], ns1[2];
        if (!PREROT && !ALIBI && !LOCAL) {
            const float4* t4 = pv.rope_pair + (size_t)(kD / 4) + 2 * u;   // position 1
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const float4 f = pv.max_position > 1 ? __ldg(t4 + v) : make_float4(1.f, 1.f, 0.f, 0.f);
                c1[v] = make_float2(f.x, f.y);
                s1[v] = make_float2(f.z, f.w);
                ns1[v] = make_float2(-f.z, -f.w);
            }
        }
        // One thread polls the stage's barrier and a named barrier releases the
        // other 127: every mbarrier update (each TMA copy's bytes) wakes its
        // pollers, and 128 pollers would take issue slots from the math roles.
        // The named barrier also makes the go / no-go decision the same for all
        // 128 threads (each reading the abort flag on its own could split them).
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
        for (int k = 0; T > 0; ++k) {
            const int st = k % kStages, ph = (k / kStages) & 1;
            if (!rot_wait(smem_u32(&bar_kfull[st]), ph)) break;
            const TileInfo& info = s_info[k & (kInfoSlots - 1)];
            if (info.j < 0) {   // no more tiles: let the MMA issuer see the sentinel
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bar_kready[st]));
                break;
            }
            const int np = info.n[p];
            // key row 16p + s, dims 4u..4u+3: 8 bytes in 16-byte unit u / 2 of each half
            uint8_t* kb = sm + kOffK + st * kKVBytes + (2 * p) * 1024 + (u & 1) * 8;
            float2 C[2], S[2];
            if (!PREROT && !ALIBI) {
                const float4* b4 = reinterpret_cast<const float4*>(sm + kOffBase + st * kBaseBytes + p * 512) + 2 * u;
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const float4 b = b4[v];   // (cos f, cos f+1, sin f, sin f+1)
                    C[v] = make_float2(b.x, b.y);
                    S[v] = make_float2(b.z, b.w);
                }
            }
#pragma unroll 1
            for (int s8 = 0; s8 < 2; ++s8) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int s = 8 * s8 + j;
                    uint2* p1 = reinterpret_cast<uint2*>(kb + s8 * 1024 + j * 128 + (((u >> 1) ^ j) << 4));
                    uint2* p2 = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(p1) + kKVChunk);
                    uint2 w1 = make_uint2(0, 0), w2 = w1;
                    if (s < np) {   // no key in this slot: zero K so that its scores stay finite
                        const uint2 a = *p1, z = *p2;
                        float x1[4] = {bf_lo(a.x), bf_hi(a.x), bf_lo(a.y), bf_hi(a.y)};
                        float x2[4] = {bf_lo(z.x), bf_hi(z.x), bf_lo(z.y), bf_hi(z.y)};
                        if (!PREROT && !ALIBI) {
#pragma unroll
                            for (int v = 0; v < 2; ++v) {
                                const float2 xa = make_float2(x1[2 * v], x1[2 * v + 1]);
                                const float2 xz = make_float2(x2[2 * v], x2[2 * v + 1]);
                                const float2 r1 = f2_sub(f2_mul(xa, C[v]), f2_mul(xz, S[v]));
                                const float2 r2 = f2_fma(xa, S[v], f2_mul(xz, C[v]));
                                x1[2 * v] = r1.x;
                                x1[2 * v + 1] = r1.y;
                                x2[2 * v] = r2.x;
                                x2[2 * v + 1] = r2.y;
                            }
                        }
                        w1 = make_uint2(pack_h2(x1[0], x1[1]), pack_h2(x1[2], x1[3]));
                        w2 = make_uint2(pack_h2(x2[0], x2[1]), pack_h2(x2[2], x2[3]));
                    }
                    *p1 = w1;
                    *p2 = w2;
                    if (!PREROT && !ALIBI && !LOCAL) {   // next slot: angle + theta
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            const float2 cc = f2_fma(C[v], c1[v], f2_mul(S[v], ns1[v]));
                            S[v] = f2_fma(S[v], c1[v], f2_mul(C[v], s1[v]));
                            C[v] = cc;
                        }
                    }
                }
            }
            // V needs no work here: pages without keys are not read (their rows
            // are outside the tensor map and read as zeros), and slots past a
            // page's valid count are zero in every page the library fills, so
            // P = 0 meets V = 0 there.
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_kready[st]));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax rows
        const int qi = (warp - 4) >> 2;            // Q tile of this warpgroup
        const int quarter = warp & 3;
        const int trow = 32 * quarter + lane;      // row within the tile = TMEM lane
        const int row = qi * kTileM + trow;        // row within the CTA
        const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);
        const uint32_t ts = tl + qi * 128;         // S_i, and P_i over its first 64 columns
        const uint32_t to = tl + 256 + qi * 128;   // O_i
        const int t_local = row / g, jh = row - t_local * g;
        const int tok = i0 + t_local;
        const int m_row = qs + tok;
        bool row_valid = t_local < ntok;
        if (row_valid && (m_row < 0 || m_row >= pv.max_position)) {
            record_error(pv.status, LAZYATTN_ERANGE);
            row_valid = false;
        }

        // Q row: rotate at m_row, scale by log2(e) times the pool's logit scale (1/sqrt(D)),
        // fp16, 128B-swizzled K-major
        {
            uint8_t* qsm = sm + kOffQ + qi * kQBytes;
            const float sc = kLog2e * pv.qk_scale;
            const __nv_bfloat16* qp_ = P.q + ((size_t)(q0 + tok) * Hq + (size_t)h * g + jh) * kD;
            const float* cs = reinterpret_cast<const float*>(pv.rope + (size_t)(row_valid ? m_row : 0) * (kD / 2));
            // The row's position-table line (512 B) is fetched into L1 while the
            // q words load; each half of the row's dims loads its q words together.
            if (!ALIBI && row_valid) {
#pragma unroll
                for (int l = 0; l < 4; ++l) asm volatile("prefetch.global.L1 [%0];" ::"l"(cs + 32 * l));
            }
#pragma unroll 1
            for (int h4 = 0; h4 < 2; ++h4) {
                uint4 qa[4], qb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int u = 4 * h4 + i;
                    qa[i] = row_valid ? __ldg(reinterpret_cast<const uint4*>(qp_ + (INTER ? 16 * u : 8 * u)))
                                      : make_uint4(0, 0, 0, 0);
                    qb[i] = row_valid ? __ldg(reinterpret_cast<const uint4*>(qp_ + (INTER ? 16 * u + 8 : 64 + 8 * u)))
                                      : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int u = 4 * h4 + i;
                    uint4 w1 = make_uint4(0, 0, 0, 0), w2 = w1;
                    if (row_valid) {
                        float x1[8], x2[8];
                        uint4 a = qa[i], b = qb[i];
                        if (INTER) deinterleave16(a, b, a, b);
                        unpack8(a, x1);
                        unpack8(b, x2);
                        float n2 = 0.f;   // input range: rotated, scaled pairs must stay finite in fp16
#pragma unroll
                        for (int v = 0; v < 8; ++v) n2 = fmaxf(n2, fmaf(x1[v], x1[v], x2[v] * x2[v]));
                        if (!(n2 * sc * sc <= kMaxPairNorm2)) record_error(pv.status, LAZYATTN_ERANGE);
                        const float4* c4 = reinterpret_cast<const float4*>(cs + 16 * u);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const float4 f = ALIBI ? make_float4(1.f, 0.f, 1.f, 0.f) : __ldg(c4 + v);
                            const float a0 = x1[2 * v], z0 = x2[2 * v], a1 = x1[2 * v + 1], z1 = x2[2 * v + 1];
                            x1[2 * v] = (a0 * f.x - z0 * f.y) * sc;
                            x2[2 * v] = (a0 * f.y + z0 * f.x) * sc;
                            x1[2 * v + 1] = (a1 * f.z - z1 * f.w) * sc;
                            x2[2 * v + 1] = (a1 * f.w + z1 * f.z) * sc;
                        }
                        w1 = pack8_h(x1);
                        w2 = pack8_h(x2);
                    }
                    *reinterpret_cast<uint4*>(qsm + sw128_offset(trow, u)) = w1;
                    *reinterpret_cast<uint4*>(qsm + kQChunk + sw128_offset(trow, u)) = w2;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_qready));
        }
        const bool active = qi == 0 || tile1;
        // ALiBi: slope of this row's query head, in the log2 domain of the scores
        const float alibi_c1 = ALIBI ? alibi_slope(h * g + jh, Hq) * kLog2e : 0.f;

        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int k = 0;
        for (; active && T > 0; ++k) {
            const int is = k & (kInfoSlots - 1);
            ok = mbar_wait(smem_u32(&bar_info[is]), (k / kInfoSlots) & 1, abort_flag);
            if (!ok) break;
            const TileInfo& info = s_info[is];
            if (info.j < 0) break;
            // a warp whose rows all see every key of the tile skips the masking
            const bool wfull = __all_sync(0xffffffffu, row_valid && m_row >= info.full_from);
            // visibility of the tile's keys to this row: bit i of visN is key
            // 32N + i (pages 2N and 2N+1 hold slots [0, lim) of their 16)
            uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
#pragma unroll
            for (int w = 0; w < 4 && !wfull; ++w) {
                uint32_t bits = 0;
#pragma unroll
                for (int hp = 0; hp < 2; ++hp) {
                    const int p = 2 * w + hp;
                    const int l = row_valid ? max(min(info.n[p], m_row - info.start[p] + 1), 0) : 0;
                    bits |= ((1u << l) - 1u) << (16 * hp);
                }
                vis[w] = bits;
            }
            ok = mbar_wait(smem_u32(&bar_sfull[qi]), k & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            // masked keys read as -inf
            auto mask64 = [&](uint32_t (&v)[64], int hh) {
                const uint32_t m0 = hh ? vis[2] : vis[0], m1 = hh ? vis[3] : vis[1];
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const uint32_t m = i < 32 ? m0 : m1;
                    v[i] = (m >> (i & 31)) & 1u ? v[i] : 0xff800000u;
                }
            };
            // ALiBi (log2 domain): key i of page q of half hh gets alibi_c1 * (start_q + i - m_row).
            // The page's start comes from the tile info (valid until this warp's P arrival).
            auto page_delta = [&](int hh, int q) { return info.start[4 * hh + q] - m_row; };
            // pass 1: row maximum over the tile
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
            // ALiBi: the reference maximum only has to bound the biased scores
            // from above (it moves by kRescaleThreshold steps anyway), so each
            // page's raw maximum takes the page's largest bias over visible keys,
            // alibi_c1 * min(start + 15 - m_row, 0) (visible keys have n <= m_row).
            float mxa = -INFINITY;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[64];
                tmem_ld64(ts + 64 * hh, v);
                if (!wfull) mask64(v, hh);
                if (ALIBI) {
                    // per page (pairs 8q .. 8q+7), two chains each
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float a = -INFINITY, c = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 8; i += 2) {
                            const int j = 8 * q + i;
                            a = fmax3(a, __uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                            c = fmax3(c, __uint_as_float(v[2 * j + 2]), __uint_as_float(v[2 * j + 3]));
                        }
                        mxa = fmax3(mxa, a + alibi_c1 * (float)min(page_delta(hh, q) + 15, 0),
                                    c + alibi_c1 * (float)min(page_delta(hh, q) + 15, 0));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        mx8[j & 7] = fmax3(mx8[j & 7], __uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                }
            }
            const float mx = ALIBI ? mxa
                                   : fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                           fmaxf(mx8[6], mx8[7]));
            float alpha = 1.f;
            if (mx > m_run + kRescaleThreshold) {
                alpha = fast_exp2(m_run - mx);   // 0 when m_run is -inf
                m_run = mx;
            }
            const float mref = (m_run == -INFINITY) ? 0.f : m_run;
            // O_i already holds tiles < k (see the header); rescale it when the
            // reference maximum moved for some row of the warp.
            if (k >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(to + 32 * c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st32(to + 32 * c, v);
                }
            }
            // pass 2: P = 2^(s - mref) as bf16 pairs over S's first 64 columns
            float2 sum4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) sum4[i] = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[64];
                tmem_ld64(ts + 64 * hh, v);
                if (!wfull) mask64(v, hh);
                uint32_t pk[32];
                if (ALIBI) {
                    // exponent = s + bias - mref; (bias - mref) of keys 2i, 2i+1 of a
                    // page stepped by 2 * alibi_c1 (masked keys stay -inf)
                    const float2 step = make_float2(2.f * alibi_c1, 2.f * alibi_c1);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float k0 = fmaf(alibi_c1, (float)page_delta(hh, q), -mref);
                        float2 w = make_float2(k0, k0 + alibi_c1);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int j = 8 * q + i;
                            const float2 d = add2(make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), w);
                            w = add2(w, step);
                            const float2 pp = make_float2(fast_exp2(d.x), fast_exp2(d.y));
                            sum4[j & 3] = add2(sum4[j & 3], pp);
                            pk[j] = pack_bf2(pp.x, pp.y);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float2 d = sub2(make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), mref);
                        const float2 pp = make_float2(fast_exp2(d.x), fast_exp2(d.y));
                        sum4[j & 3] = add2(sum4[j & 3], pp);
                        pk[j] = pack_bf2(pp.x, pp.y);
                    }
                }
                tmem_st32(ts + 32 * hh, pk);
            }
            const float2 s01 = add2(sum4[0], sum4[1]), s23 = add2(sum4[2], sum4[3]);
            const float2 s4 = add2(s01, s23);
            l_run = l_run * alpha + (s4.x + s4.y);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_pfull[qi]));
        }

        // epilogue: O / l -> bf16 rows of out; or, when the request's tiles are
        // split over several CTAs, this CTA's unnormalised O with its reference
        // maximum and sum (merged by prefill_combine_kernel)
        if (SPLIT && active) {
            if (ok && k >= 1) ok = mbar_wait(smem_u32(&bar_odone[qi]), (k - 1) & 1, abort_flag);
            tc_fence_after();
            const size_t slot = ((size_t)((r * Hkv + h) * P.qpairs + qp) * P.splits + split) * kRows + row;
            const bool keys = ok && k >= 1 && l_run > 0.f;
            if (t_local < ntok) P.part_ml[slot] = make_float2(m_run == -INFINITY ? 0.f : m_run, keys ? l_run : 0.f);
            if (k >= 1 && ok) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(to + 32 * c, v);
                    if (keys && t_local < ntok) {
                        float4* dst = reinterpret_cast<float4*>(P.part_o + slot * kD + 32 * c);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    }
                }
            }
        } else if (active) {
            if (ok && k >= 1) ok = mbar_wait(smem_u32(&bar_odone[qi]), (k - 1) & 1, abort_flag);
            tc_fence_after();
            __nv_bfloat16* op = P.out + ((size_t)(q0 + tok) * Hq + (size_t)h * g + jh) * kD;
            const float inv = (ok && l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                if (k >= 1 && ok) {
                    tmem_ld32(to + 32 * c, v);
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
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && s_abort) record_error(pv.status, LAZYATTN_EDEVICE);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge of a split prefill: thread = (row of an item, 8 dims); the partials
// with a positive sum are weighted by 2^(m_s - M), M their largest reference
// maximum (the kernel's scores are in the log2 domain).
__global__ void __launch_bounds__(256)
    prefill_combine_kernel(PoolView pv, PrefillParams P) {
    const int item = blockIdx.x, row = blockIdx.y * 16 + (threadIdx.x >> 4), d0 = (threadIdx.x & 15) * 8;
    const int g = P.g, Hkv = pv.hkv;
    const int qp = item % P.qpairs, h = (item / P.qpairs) % Hkv, r = item / (P.qpairs * Hkv);
    const int TQ = kRows / g;
    const int q0 = P.q_offsets[r], q1 = P.q_offsets[r + 1];
    const int tok = qp * TQ + row / g, jh = row % g;
    if (tok >= q1 - q0) return;
    const size_t base = (size_t)item * P.splits * kRows + row;
    float M = -INFINITY;
    for (int sp = 0; sp < P.splits; ++sp) {
        const float2 x = __ldcg(&P.part_ml[base + (size_t)sp * kRows]);
        if (x.y > 0.f) M = fmaxf(M, x.x);
    }
    float L = 0.f, a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.f;
    if (M != -INFINITY) {
        for (int sp = 0; sp < P.splits; ++sp) {
            const size_t slot = base + (size_t)sp * kRows;
            const float2 x = __ldcg(&P.part_ml[slot]);
            if (!(x.y > 0.f)) continue;
            const float w = fast_exp2(x.x - M);
            L += x.y * w;
            const float4* src = reinterpret_cast<const float4*>(P.part_o + slot * kD + d0);
            const float4 s0 = __ldcg(src), s1 = __ldcg(src + 1);
            a[0] += s0.x * w; a[1] += s0.y * w; a[2] += s0.z * w; a[3] += s0.w * w;
            a[4] += s1.x * w; a[5] += s1.y * w; a[6] += s1.z * w; a[7] += s1.w * w;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(P.out + ((size_t)(q0 + tok) * pv.hq + (size_t)h * g + jh) * kD + d0);
    *dst = make_uint4(pack_bf2(a[0] * inv, a[1] * inv), pack_bf2(a[2] * inv, a[3] * inv),
                      pack_bf2(a[4] * inv, a[5] * inv), pack_bf2(a[6] * inv, a[7] * inv));
}

}  // namespace

using PrefillKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                               const CUtensorMap, const CUtensorMap, const CUtensorMap, PoolView, PrefillParams);

// The instantiation for a pool and a batch: key layout and pairing of the pool,
// pre-rotated pages of the batch.
template <bool SPLIT>
PrefillKernel prefill_kernel_variant(bool prerot, bool local, bool inter, bool alibi) {
    if (alibi) return prefill_tc_kernel<false, false, false, true, SPLIT>;
    if (local)
        return inter ? prefill_tc_kernel<false, true, true, false, SPLIT> : prefill_tc_kernel<false, true, false, false, SPLIT>;
    if (prerot)
        return inter ? prefill_tc_kernel<true, false, true, false, SPLIT> : prefill_tc_kernel<true, false, false, false, SPLIT>;
    return inter ? prefill_tc_kernel<false, false, true, false, SPLIT> : prefill_tc_kernel<false, false, false, false, SPLIT>;
}

PrefillKernel prefill_kernel_for(bool prerot, bool local, bool inter, bool alibi, bool split) {
    return split ? prefill_kernel_variant<true>(prerot, local, inter, alibi)
                 : prefill_kernel_variant<false>(prerot, local, inter, alibi);
}

int prefill_init() {
    for (int sp = 0; sp < 2; ++sp)
        for (int i = 0; i < 9; ++i) {
            if (i < 8 && (i & 1) && (i & 2)) continue;   // pre-rotated pages are never doc-local
            PrefillKernel k = i == 8 ? prefill_kernel_for(false, false, false, true, sp)
                                     : prefill_kernel_for(i & 1, i & 2, i & 4, false, sp);
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
                return LAZYATTN_ECUDA;
        }
    return LAZYATTN_OK;
}

// Split count of a prefill over its KV tiles. A CTA per (request, KV head,
// query pair) runs its tiles at a steady rate after a start-up and drain of
// about five tiles' time; when such CTAs fill few waves of the GPU, the last
// wave runs part-empty, and splitting every CTA's tiles s ways trades that for
// s - 1 more start-ups per item and a merge of the partials (written, then
// read: about 6 MB per tile's time, merge launch included). Both constants are
// fitted to GB300 timings of the TTFT-sweep batches at s = 1..4. The model picks
// the s in 1..4 with the least estimated time; shares stay at least 8 tiles.
int prefill_splits(const lazyattn_pool& p, const lazyattn_batch& b) {
    const int g = p.d.n_q_heads / p.d.n_kv_heads;
    if (p.d.dtype != LAZYATTN_BF16 || p.d.head_dim != kD || kRows % g != 0 || b.max_q_len < 1) return 1;
    const int64_t TQ = kRows / g;
    const int64_t items = (int64_t)b.num_requests * p.d.n_kv_heads * ((b.max_q_len + TQ - 1) / TQ);
    const int64_t T = ((int64_t)b.max_entries + kPagesPerTile - 1) / kPagesPerTile;
    const int64_t sms = p.sm_count > 0 ? p.sm_count : 1;
    const double merge_bytes_per_tile = 6e6, startup_tiles = 5.0;
    int best = 1;
    double best_cost = 0.0;
    for (int s = 1; s <= 4; ++s) {
        if (s > 1 && T / s < 8) break;
        const int64_t ctas = items * s;
        const double waves = (double)((ctas + sms - 1) / sms);
        double cost = waves * ((double)((T + s - 1) / s) + startup_tiles);
        if (s > 1) cost += (double)ctas * kRows * (kD * 4 + 8) * 2.0 / merge_bytes_per_tile;   // written + read
        if (s == 1 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

size_t prefill_ws_bytes(const lazyattn_pool& p, const lazyattn_batch& b, int splits) {
    if (splits <= 1) return 0;
    const int g = p.d.n_q_heads / p.d.n_kv_heads;
    const size_t TQ = kRows / g;
    const size_t items = (size_t)b.num_requests * p.d.n_kv_heads * ((b.max_q_len + TQ - 1) / TQ);
    const size_t slots = items * splits * kRows;
    return ((slots * kD * sizeof(float) + 255) & ~size_t(255)) + slots * sizeof(float2);
}

int launch_prefill_bf16(const lazyattn_pool& p, const lazyattn_batch& b, const __nv_bfloat16* q,
                        __nv_bfloat16* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
    const int g = p.d.n_q_heads / p.d.n_kv_heads;
    if (p.d.head_dim != kD || kRows % g != 0) return LAZYATTN_EINVAL;
    if (!p.have_maps) return LAZYATTN_ECUDA;
    if (b.max_q_len < 1) return LAZYATTN_OK;
    const uint64_t rows = (uint64_t)p.d.num_pages * (uint64_t)p.d.n_kv_heads * kPage;
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
    P.entry_delta = b.entry_delta;
    P.row_blocks = p.have_rmap ? p.d.max_position / kPage : 0;
    const int TQ = kRows / g;
    P.qpairs = (b.max_q_len + TQ - 1) / TQ;
    P.splits = prefill_splits(p, b);
    P.part_o = nullptr;
    P.part_ml = nullptr;
    if (P.splits > 1) {
        const size_t need = prefill_ws_bytes(p, b, P.splits);
        if (ws && ws_bytes >= need && !(reinterpret_cast<uintptr_t>(ws) & 255u)) {
            const size_t slots = (size_t)b.num_requests * p.d.n_kv_heads * P.qpairs * P.splits * kRows;
            P.part_o = static_cast<float*>(ws);
            P.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) +
                                                  ((slots * kD * sizeof(float) + 255) & ~size_t(255)));
        } else {
            P.splits = 1;   // no room for the partials: one CTA per item
        }
    }
    dim3 grid(P.qpairs * P.splits, p.d.n_kv_heads, b.num_requests);
    auto kern = prefill_kernel_for((b.flags & LAZYATTN_KEYS_PREROTATED) != 0,
                                   p.d.key_storage == LAZYATTN_KEYS_DOC_LOCAL, p.d.rope_interleaved != 0,
                                   p.d.position_encoding == LAZYATTN_POS_ALIBI, P.splits > 1);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(p.kmap, p.vmap, p.kmap4, p.vmap4, p.kmap8, p.vmap8, p.rmap, p.view(),
                                                 P);
    if (cudaGetLastError() != cudaSuccess) return LAZYATTN_ECUDA;
    if (P.splits > 1) {
        prefill_combine_kernel<<<dim3(P.qpairs * p.d.n_kv_heads * b.num_requests, kRows / 16), 256, 0, stream>>>(
            p.view(), P);
        if (cudaGetLastError() != cudaSuccess) return LAZYATTN_ECUDA;
    }
    return LAZYATTN_OK;
}

}  // namespace lazyattn
