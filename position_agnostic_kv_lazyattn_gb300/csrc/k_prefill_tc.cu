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
// rotation serve 256 rows of the group. Tiles of 64 keys (4 pages) stream
// through a 3-stage ring. Roles (16 warps = 4 warpgroups):
//   warps 0, 2    TMA producers, K ring and V ring: per tile 4 pages x two
//                 64-dim boxes (128B swizzle); with K, each page's row
//                 (cos, sin)(start * theta) of the position table (bulk copy)
//   warp 1        TMEM owner and single-thread UMMA issuer, per tile:
//                 S_i = Q_i K^T (fp16, 128x64x128) for both Q tiles, then
//                 O_i += P_i V of the previous tile (bf16, 128x128x64)
//   warps 4-7     softmax of Q tile 0; warps 8-11 softmax of Q tile 1: one row
//                 per thread (TMEM lane), causal + validity mask on logical
//                 positions, online softmax in the log2 domain with lazy
//                 rescaling of O (only when the row max grows by > 8), P as bf16
//                 to shared memory; final normalisation and store
//   warps 12-15   K rotation: half a key row per thread; cos/sin of start+slot by
//                 angle addition of the page's row and a 16-row slot table kept
//                 in shared memory; written back in place as fp16
// S is double-buffered per Q tile in TMEM (4 x 64 columns) next to O (2 x 128).
// Tiles whose keys are all masked for every row of the CTA (past the causal
// edge, or empty entries) are skipped. Only the producer reads the block
// table: with each stage it publishes the tile's page starts and token counts
// in shared memory (before arriving on the stage's barrier), and after the last
// tile a sentinel stage, so the consumer roles never touch global memory inside
// the tile loop. Every wait is
// bounded; a timeout raises an abort flag that all roles honour, drains
// in-flight copies and MMAs, frees TMEM and records LAZYATTN_EDEVICE.
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
constexpr int kN = 64;                             // keys per K/V tile
constexpr int kPagesPerTile = kN / kPage;          // 4
constexpr int kStages = 3;
constexpr int kThreads = 512;
constexpr int kQBytes = kTileM * kD * 2;           // 32 KB
constexpr int kQChunk = kTileM * 128;              // 16 KB (64 dims)
constexpr int kKVBytes = kN * kD * 2;              // 16 KB
constexpr int kKVChunk = kN * 128;                 // 8 KB (64 dims)
constexpr int kBaseBytes = kPagesPerTile * 512;    // 4 position-table rows
constexpr int kPBytes = kTileM * kN * 2;           // 16 KB
constexpr int kSlotRow = 528;                      // 512 B + 16 B pad (conflict-free column reads)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQTiles * kQBytes;
constexpr int kOffV = kOffK + kStages * kKVBytes;
constexpr int kOffP = kOffV + kStages * kKVBytes;
constexpr int kOffBase = kOffP + kQTiles * kPBytes;
constexpr int kOffSlot = kOffBase + kStages * kBaseBytes;
constexpr int kSmemUsed = kOffSlot + kPage * kSlotRow;
constexpr int kSmemBytes = kSmemUsed + 1024;       // + alignment slack
constexpr uint32_t kTmemCols = 512;                // S[i][b] at i*128 + b*64; O[i] at 256 + i*128
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;          // log2 units

static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles need 1 KB alignment");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// What the producer tells the consumers about the tile in a stage.
struct TileInfo {
    int j;                        // tile index, -1: no more tiles
    int start[kPagesPerTile];     // logical position of slot 0 of each page
    int n[kPagesPerTile];         // keys in each page (0: none / unusable)
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

// Entry check shared by every role so that all of them agree on which slots
// hold keys: page in range and positions inside the table.
__device__ __forceinline__ int usable_tokens(const PoolView& pv, uint64_t e) {
    const int n = entry_nvalid(e);
    if (n == 0) return 0;
    if (entry_page(e) >= (uint32_t)pv.num_pages || n > kPage || entry_start(e) + n > pv.max_position) return -1;
    return n;
}

// A tile is processed iff one of its pages holds a key at a position <= the
// largest query position of the CTA. Every role evaluates this identically.
__device__ __forceinline__ bool tile_live(const PoolView& pv, const uint64_t* entries, int e0, int e1, int j,
                                          int m_hi) {
    bool live = false;
#pragma unroll
    for (int p = 0; p < kPagesPerTile; ++p) {
        const int idx = e0 + j * kPagesPerTile + p;
        if (idx < e1) {
            const uint64_t e = entries[idx];
            live = live || (usable_tokens(pv, e) > 0 && entry_start(e) <= m_hi);
        }
    }
    return live;
}

template <bool PREROT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, PoolView pv,
                      PrefillParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    __shared__ uint64_t bar_kfull[kStages], bar_kempty[kStages], bar_vfull[kStages], bar_vempty[kStages];
    __shared__ uint64_t bar_kready[kStages];
    __shared__ uint64_t bar_sfull[kQTiles][2], bar_sfree[kQTiles][2], bar_pfull[kQTiles], bar_odone[kQTiles];
    __shared__ uint64_t bar_qready, bar_drain;
    __shared__ TileInfo s_info[kStages];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int qp = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
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
    const int T = e1 > e0 ? (e1 - e0 + kPagesPerTile - 1) / kPagesPerTile : 0;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_kfull[s]), 1);
            mbar_init(smem_u32(&bar_kempty[s]), 1);
            mbar_init(smem_u32(&bar_vfull[s]), 1);
            mbar_init(smem_u32(&bar_vempty[s]), 1);
            mbar_init(smem_u32(&bar_kready[s]), 128);
        }
        for (int i = 0; i < kQTiles; ++i) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&bar_sfull[i][b]), 1);
                mbar_init(smem_u32(&bar_sfree[i][b]), 128);
            }
            mbar_init(smem_u32(&bar_pfull[i]), 128);
            mbar_init(smem_u32(&bar_odone[i]), 1);
        }
        mbar_init(smem_u32(&bar_qready), kQTiles * 128);
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

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ TMA producers
        // Warp 0 streams K tiles (with the pages' position-table rows and the
        // tile info), warp 2 streams V tiles, each through its own ring: a K
        // stage is reused once the tile's QK MMAs are done, a V stage once its PV
        // MMAs are, so both loads are requested several tiles ahead.
        const bool is_k = warp == 0;
        if (lane == 0 && T > 0) {
            uint64_t* full = is_k ? bar_kfull : bar_vfull;
            uint64_t* empty = is_k ? bar_kempty : bar_vempty;
            const CUtensorMap* map = is_k ? &kmap : &vmap;
            const int off = is_k ? kOffK : kOffV;
            int last_k[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) last_k[s] = -1;
            int k = 0;
            bool ok = true;
            for (int j = 0; j <= T; ++j) {
                if (j < T && !tile_live(pv, P.entries, e0, e1, j, m_hi)) continue;
                if (j == T && !is_k) break;
                const int st = k % kStages;
                if (k >= kStages && !mbar_wait(smem_u32(&empty[st]), ((k / kStages) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&full[st]);
                TileInfo& info = s_info[st];
                if (j == T) {   // sentinel: no more tiles
                    info.j = -1;
                    mbar_arrive(fb);
                    break;
                }
                const uint32_t ds = smem_u32(sm + off + st * kKVBytes);
                const uint32_t bs = smem_u32(sm + kOffBase + st * kBaseBytes);
                int ys[kPagesPerTile];
                const float2* bases[kPagesPerTile];
                for (int p = 0; p < kPagesPerTile; ++p) {
                    const int idx = e0 + j * kPagesPerTile + p;
                    int y = P.oob_row, n = 0, st0 = 0;
                    const float2* base = pv.rope;
                    if (idx < e1) {
                        const uint64_t e = P.entries[idx];
                        n = usable_tokens(pv, e);
                        st0 = entry_start(e);
                        if (n < 0 && is_k) record_error(pv.status, LAZYATTN_ERANGE);
                        if (n > 0) {
                            y = ((int)entry_page(e) * Hkv + h) * kPage;
                            base = pv.rope + (size_t)st0 * (kD / 2);
                        }
                    }
                    if (is_k) {
                        info.start[p] = st0;
                        info.n[p] = max(n, 0);
                    }
                    ys[p] = y;
                    bases[p] = base;
                }
                if (is_k) info.j = j;
                // arrive before the copies: releases the info writes to the waiters
                mbar_arrive_expect_tx(fb, is_k ? kKVBytes + kBaseBytes : kKVBytes);
                for (int p = 0; p < kPagesPerTile; ++p) {
                    tma_load_2d(ds + p * 2048, map, 0, ys[p], fb);
                    tma_load_2d(ds + kKVChunk + p * 2048, map, 64, ys[p], fb);
                    if (is_k) bulk_load(bs + p * 512, bases[p], 512, fb);
                }
                last_k[st] = k;
                ++k;
            }
            if (!ok) *abort_flag = 1;
            if (*abort_flag) {   // let issued copies land before the CTA's smem is released
                volatile int never = 0;
                for (int s = 0; s < kStages; ++s)
                    if (last_k[s] >= 0) mbar_wait(smem_u32(&full[s]), (last_k[s] / kStages) & 1, &never);
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
            // Q tiles, P tiles and ring stages are evenly spaced: index * stride.
            const uint64_t dq0 = sdesc_sw128(smem_u32(sm + kOffQ), 16, 1024);
            const uint64_t dp0 = sdesc_sw128(smem_u32(sm + kOffP), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(smem_u32(sm + kOffK), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(sm + kOffV), kKVChunk, 1024);
            auto issue_qk = [&](int i, int st, int b) {
                const uint64_t a0 = dq0 + (uint64_t)(i * (kQBytes >> 4)), b0 = dk0 + (uint64_t)(st * (kKVBytes >> 4));
                const uint32_t d = tmem + i * 128 + b * kN;
#pragma unroll
                for (int t = 0; t < kD / 16; ++t) {
                    const uint64_t oa = (uint64_t)(((t >> 2) * kQChunk + (t & 3) * 32) >> 4);
                    const uint64_t ob = (uint64_t)(((t >> 2) * kKVChunk + (t & 3) * 32) >> 4);
                    umma_f16(d, a0 + oa, b0 + ob, idqk, t > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int i, int st, uint32_t first) {
                const uint64_t a0 = dp0 + (uint64_t)(i * (kPBytes >> 4)), b0 = dv0 + (uint64_t)(st * (kKVBytes >> 4));
                const uint32_t d = tmem + 256 + i * 128;
#pragma unroll
                for (int t = 0; t < kN / 16; ++t)
                    umma_f16(d, a0 + (uint64_t)(t * 2), b0 + (uint64_t)(t * 128), idpv, (t > 0 || !first) ? 1u : 0u);
            };
            bool ok = T > 0 && mbar_wait(smem_u32(&bar_qready), 0, abort_flag);
            int k = 0;
            for (; ok;) {
                const int st = k % kStages, b = k & 1;
                ok = mbar_wait(smem_u32(&bar_kfull[st]), (k / kStages) & 1, abort_flag);
                if (!ok || s_info[st].j < 0) break;
                ok = mbar_wait(smem_u32(&bar_kready[st]), (k / kStages) & 1, abort_flag);
                if (!ok) break;
                for (int i = 0; ok && i < nt; ++i) {
                    if (k >= 2) ok = mbar_wait(smem_u32(&bar_sfree[i][b]), ((k >> 1) - 1) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(i, st, b);
                    umma_commit(smem_u32(&bar_sfull[i][b]));
                }
                if (!ok) break;
                umma_commit(smem_u32(&bar_kempty[st]));   // K stage free once these QK MMAs finish
                if (k >= 1) {   // P V of the previous tile
                    const int pst = (k - 1) % kStages;
                    ok = mbar_wait(smem_u32(&bar_vfull[pst]), ((k - 1) / kStages) & 1, abort_flag);
                    for (int i = 0; ok && i < nt; ++i) {
                        ok = mbar_wait(smem_u32(&bar_pfull[i]), (k - 1) & 1, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(i, pst, k == 1);
                        umma_commit(smem_u32(&bar_odone[i]));
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&bar_vempty[pst]));
                }
                ++k;
            }
            if (ok && k >= 1) {   // P V of the last tile
                const int pst = (k - 1) % kStages;
                ok = mbar_wait(smem_u32(&bar_vfull[pst]), ((k - 1) / kStages) & 1, abort_flag);
                for (int i = 0; ok && i < nt; ++i) {
                    ok = mbar_wait(smem_u32(&bar_pfull[i]), (k - 1) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(i, pst, k == 1);
                    umma_commit(smem_u32(&bar_odone[i]));
                }
                umma_commit(smem_u32(&bar_vempty[pst]));
            }
            // every issued MMA has finished before TMEM / smem are released
            umma_commit(smem_u32(&bar_drain));
            volatile int never = 0;
            mbar_wait(smem_u32(&bar_drain), 0, &never);
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ K rotation
        const int rt = threadIdx.x - 384;
        uint8_t* slot_tab = sm + kOffSlot;   // row t: (cos, sin)(t * theta_i)
        for (int i = rt; i < kPage * 32; i += 128) {
            const int t = i >> 5, f4 = i & 31;
            const float4 v = t < pv.max_position ? __ldg(reinterpret_cast<const float4*>(pv.rope) + t * 32 + f4)
                                                 : make_float4(1.f, 0.f, 1.f, 0.f);
            *reinterpret_cast<float4*>(slot_tab + t * kSlotRow + f4 * 16) = v;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");   // slot table complete (rotation warps only)
        const int kr = rt >> 1, hf = rt & 1;              // key row of the tile, half of its units
        const int slot = kr & 15;
        for (int k = 0; T > 0; ++k) {
            const int st = k % kStages;
            if (!mbar_wait(smem_u32(&bar_kfull[st]), (k / kStages) & 1, abort_flag)) break;
            const TileInfo& info = s_info[st];
            if (info.j < 0) break;
            const bool valid = slot < info.n[kr >> 4];
            bool partial = false;   // a page with some, but not all, slots holding keys
#pragma unroll
            for (int p = 0; p < kPagesPerTile; ++p) partial = partial || (info.n[p] > 0 && info.n[p] < kPage);
            uint8_t* kb = sm + kOffK + st * kKVBytes;
            uint8_t* vb = sm + kOffV + st * kKVBytes;
            if (valid) {
                const float4* base = reinterpret_cast<const float4*>(sm + kOffBase + st * kBaseBytes + (kr >> 4) * 512);
                const float4* sl = reinterpret_cast<const float4*>(slot_tab + slot * kSlotRow);
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const int u = 4 * hf + uu;
                    uint4* p1 = reinterpret_cast<uint4*>(kb + sw128_offset(kr, u));
                    uint4* p2 = reinterpret_cast<uint4*>(kb + kKVChunk + sw128_offset(kr, u));
                    float x1[8], x2[8];
                    unpack8(*p1, x1);
                    unpack8(*p2, x2);
                    if (!PREROT) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {   // frequencies 8u + 2v, 8u + 2v + 1
                            const float4 b4 = base[4 * u + v], s4 = sl[4 * u + v];
                            const float c0 = b4.x * s4.x - b4.y * s4.y, n0 = b4.y * s4.x + b4.x * s4.y;
                            const float c1 = b4.z * s4.z - b4.w * s4.w, n1 = b4.w * s4.z + b4.z * s4.w;
                            const float a0 = x1[2 * v], z0 = x2[2 * v], a1 = x1[2 * v + 1], z1 = x2[2 * v + 1];
                            x1[2 * v] = a0 * c0 - z0 * n0;
                            x2[2 * v] = a0 * n0 + z0 * c0;
                            x1[2 * v + 1] = a1 * c1 - z1 * n1;
                            x2[2 * v + 1] = a1 * n1 + z1 * c1;
                        }
                    }
                    *p1 = pack8_h(x1);
                    *p2 = pack8_h(x2);
                }
            } else {   // no key in this slot: zero K so that its scores stay finite
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const int u = 4 * hf + uu;
                    *reinterpret_cast<uint4*>(kb + sw128_offset(kr, u)) = z;
                    *reinterpret_cast<uint4*>(kb + kKVChunk + sw128_offset(kr, u)) = z;
                }
            }
            if (partial) {   // stale slots of a partly filled page: zero V too (0 * NaN would be NaN)
                if (!mbar_wait(smem_u32(&bar_vfull[st]), (k / kStages) & 1, abort_flag)) break;
                if (!valid) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        const int u = 4 * hf + uu;
                        *reinterpret_cast<uint4*>(vb + sw128_offset(kr, u)) = z;
                        *reinterpret_cast<uint4*>(vb + kKVChunk + sw128_offset(kr, u)) = z;
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_kready[st]));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax rows
        const int qi = (warp - 4) >> 2;            // Q tile of this warpgroup
        const int quarter = warp & 3;
        const int trow = 32 * quarter + lane;      // row within the tile = TMEM lane
        const int row = qi * kTileM + trow;        // row within the CTA
        const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);
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
            uint8_t* qsm = sm + kOffQ + qi * kQBytes;
            const float sc = kLog2e * rsqrtf((float)kD);
            const __nv_bfloat16* qp_ = P.q + ((size_t)(q0 + tok) * Hq + (size_t)h * g + jh) * kD;
            const float* cs = reinterpret_cast<const float*>(pv.rope + (size_t)(row_valid ? m_row : 0) * (kD / 2));
#pragma unroll 2
            for (int u = 0; u < 8; ++u) {
                uint4 w1 = make_uint4(0, 0, 0, 0), w2 = w1;
                if (row_valid) {
                    float x1[8], x2[8];
                    unpack8(__ldg(reinterpret_cast<const uint4*>(qp_ + 8 * u)), x1);
                    unpack8(__ldg(reinterpret_cast<const uint4*>(qp_ + 64 + 8 * u)), x2);
                    const float4* c4 = reinterpret_cast<const float4*>(cs + 16 * u);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float4 f = __ldg(c4 + v);
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
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_qready));
        }
        const bool active = qi == 0 || tile1;

        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int k = 0;
        for (; active && T > 0; ++k) {
            const int st = k % kStages, b = k & 1;
            ok = mbar_wait(smem_u32(&bar_kfull[st]), (k / kStages) & 1, abort_flag);
            if (!ok) break;
            const TileInfo& info = s_info[st];
            if (info.j < 0) break;
            // which keys of the tile this row may see
            int kstart[kPagesPerTile], kn[kPagesPerTile];
            bool full = row_valid;
#pragma unroll
            for (int p = 0; p < kPagesPerTile; ++p) {
                kstart[p] = info.start[p];
                kn[p] = info.n[p];
                full = full && (kn[p] == kPage) && (kstart[p] + kPage - 1 <= m_row);
            }
            ok = mbar_wait(smem_u32(&bar_sfull[qi][b]), (k >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            float s[kN];
#pragma unroll
            for (int c = 0; c < kN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tl + qi * 128 + b * kN + 32 * c, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(v[i]);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sfree[qi][b]));
            if (!full) {
#pragma unroll
                for (int kk = 0; kk < kN; ++kk) {
                    const int p = kk >> 4, sl = kk & 15;
                    const bool vis = row_valid && sl < kn[p] && kstart[p] + sl <= m_row;
                    s[kk] = vis ? s[kk] : -INFINITY;
                }
            }
            float mx8[8];   // eight independent chains instead of one 64-long one
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mx8[kk] = s[kk];
#pragma unroll
            for (int kk = 8; kk < kN; ++kk) mx8[kk & 7] = fmaxf(mx8[kk & 7], s[kk]);
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            float alpha = 1.f;
            if (mx > m_run + kRescaleThreshold) {
                alpha = fast_exp2(m_run - mx);   // 0 when m_run is -inf
                m_run = mx;
            }
            const float mref = (m_run == -INFINITY) ? 0.f : m_run;
            float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pk[kN / 2];
#pragma unroll
            for (int kk = 0; kk < kN; kk += 2) {
                const float p0 = fast_exp2(s[kk] - mref), p1 = fast_exp2(s[kk + 1] - mref);
                sum8[(kk >> 1) & 7] += p0 + p1;
                pk[kk / 2] = pack_bf2(p0, p1);
            }
            const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
            l_run = l_run * alpha + sum;
            if (k >= 1) {
                ok = mbar_wait(smem_u32(&bar_odone[qi]), (k - 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tl + 256 + qi * 128 + 32 * c, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        tmem_st32(tl + 256 + qi * 128 + 32 * c, v);
                    }
                    tmem_wait_st();
                }
            }
            uint8_t* ps = sm + kOffP + qi * kPBytes;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4*>(ps + sw128_offset(trow, u)) =
                    make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_pfull[qi]));
        }

        // epilogue: O / l -> bf16 rows of out
        if (active) {
            if (ok && k >= 1) ok = mbar_wait(smem_u32(&bar_odone[qi]), (k - 1) & 1, abort_flag);
            tc_fence_after();
            __nv_bfloat16* op = P.out + ((size_t)(q0 + tok) * Hq + (size_t)h * g + jh) * kD;
            const float inv = (ok && l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                if (k >= 1 && ok) {
                    tmem_ld32(tl + 256 + qi * 128 + 32 * c, v);
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

}  // namespace

int prefill_init() {
    if (cudaFuncSetAttribute(prefill_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(prefill_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess)
        return LAZYATTN_ECUDA;
    return LAZYATTN_OK;
}

int launch_prefill_bf16(const lazyattn_pool& p, const lazyattn_batch& b, const __nv_bfloat16* q,
                        __nv_bfloat16* out, cudaStream_t stream) {
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
    const int TQ = kRows / g;
    dim3 grid((b.max_q_len + TQ - 1) / TQ, p.d.n_kv_heads, b.num_requests);
    auto kern = (b.flags & LAZYATTN_KEYS_PREROTATED) ? prefill_tc_kernel<true> : prefill_tc_kernel<false>;
    kern<<<grid, kThreads, kSmemBytes, stream>>>(p.kmap, p.vmap, p.view(), P);
    return cudaGetLastError() == cudaSuccess ? LAZYATTN_OK : LAZYATTN_ECUDA;
}

}  // namespace lazyattn
