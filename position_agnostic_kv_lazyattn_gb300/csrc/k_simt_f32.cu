// fp32 attention on CUDA cores: one warp per (query row, query head).
//
// Serves the fp32 workload, where tensor-core inputs (tf32 at best) cannot hold
// a 1e-4 tolerance. Each lane owns head dimensions {lane + 32 j}; with
// rotate-half pairing (d, d + D/2) both members of a pair sit in the same lane,
// so RoPE is applied to every key in registers at its own logical position.
#include "internal.h"

namespace lazyattn {

namespace {

template <int D, bool PREROT>
__global__ void attention_f32_kernel(PoolView pv, const uint64_t* __restrict__ entries,
                                     const int32_t* __restrict__ entry_offsets,
                                     const int32_t* __restrict__ q_offsets, const int32_t* __restrict__ q_start,
                                     const int32_t* __restrict__ decode_qpos, int32_t total_q,
                                     const float* __restrict__ q, float* __restrict__ out) {
    constexpr int J = D / 32;          // dims per lane
    constexpr int HALF = D / 2;
    const int lane = threadIdx.x;
    const int r = blockIdx.z;
    const int h = blockIdx.y;
    const int i = blockIdx.x;
    const int g = pv.hq / pv.hkv;
    const int kvh = h / g;

    int row, m;
    if (decode_qpos) {
        row = r;
        m = decode_qpos[r];
    } else {
        const int q0 = q_offsets[r], q1 = q_offsets[r + 1];
        if (i >= q1 - q0) return;
        row = q0 + i;
        if (row >= total_q || q1 > total_q) {
            record_error(pv.status, LAZYATTN_ERANGE);
            return;
        }
        m = q_start[r] + i;
    }
    float* o = out + ((size_t)row * pv.hq + h) * D;
    if (m < 0 || m >= pv.max_position) {
        if (m >= pv.max_position) record_error(pv.status, LAZYATTN_ERANGE);
        for (int j = 0; j < J; ++j) o[lane + 32 * j] = 0.f;
        return;
    }

    // q rotated at its own position m, pre-scaled by the logit scale (1/sqrt(D))
    float qr[J];
    {
        const float* qp = q + ((size_t)row * pv.hq + h) * D;
        const float sc = pv.qk_scale;
#pragma unroll
        for (int j = 0; j < J / 2; ++j) {
            const int d = lane + 32 * j;
            const float2 cs = pv.rope[(size_t)m * HALF + d];
            const float a = qp[d], b = qp[d + HALF];
            qr[j] = (a * cs.x - b * cs.y) * sc;
            qr[j + J / 2] = (a * cs.y + b * cs.x) * sc;
        }
    }

    const float* kpool = static_cast<const float*>(pv.k_pool);
    const float* vpool = static_cast<const float*>(pv.v_pool);
    float mx = -INFINITY, l = 0.f, acc[J];
#pragma unroll
    for (int j = 0; j < J; ++j) acc[j] = 0.f;

    const int e0 = entry_offsets[r], e1 = entry_offsets[r + 1];
    for (int ei = e0; ei < e1; ++ei) {
        const uint64_t e = entries[ei];
        const int n = entry_nvalid(e);
        if (n == 0 || !entry_ok(pv, e)) continue;
        const int start = entry_start(e);
        const size_t base = ((size_t)entry_page(e) * pv.hkv + kvh) * kPage * D;
        for (int s = 0; s < n; ++s) {
            const int pos = start + s;
            if (pos > m) break;
            const float* kr = kpool + base + (size_t)s * D;
            const float* vr = vpool + base + (size_t)s * D;
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < J / 2; ++j) {
                const int d = lane + 32 * j;
                float a = kr[d], b = kr[d + HALF];
                if (!PREROT) {
                    const float2 cs = pv.rope[(size_t)pos * HALF + d];
                    const float ra = a * cs.x - b * cs.y;
                    const float rb = a * cs.y + b * cs.x;
                    a = ra;
                    b = rb;
                }
                dot = fmaf(qr[j], a, dot);
                dot = fmaf(qr[j + J / 2], b, dot);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float mn = fmaxf(mx, dot);
            const float corr = __expf(mx - mn);
            const float p = __expf(dot - mn);
            l = l * corr + p;
#pragma unroll
            for (int j = 0; j < J / 2; ++j) {
                const int d = lane + 32 * j;
                acc[j] = acc[j] * corr + p * vr[d];
                acc[j + J / 2] = acc[j + J / 2] * corr + p * vr[d + HALF];
            }
            mx = mn;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int j = 0; j < J / 2; ++j) {
        const int d = lane + 32 * j;
        o[d] = acc[j] * inv;
        o[d + HALF] = acc[j + J / 2] * inv;
    }
}

}  // namespace

int launch_attention_f32(const lazyattn_pool& p, const lazyattn_batch& b, const float* q, float* out,
                         const int32_t* decode_qpos, cudaStream_t stream) {
    const bool pre = (b.flags & LAZYATTN_KEYS_PREROTATED) != 0;
    const int rows = decode_qpos ? 1 : b.max_q_len;
    if (rows < 1) return LAZYATTN_OK;
    dim3 grid(rows, p.d.n_q_heads, b.num_requests);
    const PoolView pv = p.view();
    const int total_q = decode_qpos ? b.num_requests : b.total_q;
    if (p.d.head_dim == 64) {
        auto k = pre ? attention_f32_kernel<64, true> : attention_f32_kernel<64, false>;
        k<<<grid, 32, 0, stream>>>(pv, b.entries, b.entry_offsets, b.q_offsets, b.q_start, decode_qpos, total_q, q,
                                   out);
    } else {
        auto k = pre ? attention_f32_kernel<128, true> : attention_f32_kernel<128, false>;
        k<<<grid, 32, 0, stream>>>(pv, b.entries, b.entry_offsets, b.q_offsets, b.q_start, decode_qpos, total_q, q,
                                   out);
    }
    return cudaGetLastError() == cudaSuccess ? LAZYATTN_OK : LAZYATTN_ECUDA;
}

}  // namespace lazyattn
