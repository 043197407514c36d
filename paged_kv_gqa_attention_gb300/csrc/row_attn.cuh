// Warp-per-row attention over packed segments (CUDA cores).
//
// One warp computes the outputs of the GROUP query heads that share KV head
// g for one packed row t, with an fp32 online softmax over the row's visible
// keys read straight from the packed k/v (L2-resident for these sizes).
// Visible keys: the row's own segment [cu[s], cu[s+1]) when CAUSAL is false
// (windowed encoder attention), its prefix [cu[s], t] when CAUSAL is true
// (causal prefill).  Lane l owns dims [l*E, l*E + E), E = D / 32.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace qa {

struct RowAttnArgs {
    const uint16_t *q;  // [T][hq][D]
    const uint16_t *k;  // [T][hkv][D]
    const uint16_t *v;
    const int32_t *cu;  // [n_seg + 1]
    uint16_t *out;      // [T][hq][D]
    int n_seg, total, hkv;
    float scale_log2;
};

template <int E>
__device__ __forceinline__ void load_bf16(const uint16_t *p, float (&x)[E]) {
    if constexpr (E == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(p);
        x[0] = bf16lo(w.x);
        x[1] = bf16hi(w.x);
        x[2] = bf16lo(w.y);
        x[3] = bf16hi(w.y);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
        x[0] = bf16lo(w);
        x[1] = bf16hi(w);
    }
}

template <int E>
__device__ __forceinline__ void store_bf16(uint16_t *p, const float (&x)[E]) {
    if constexpr (E == 4) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    } else {
        *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(x[0], x[1]);
    }
}

template <int D, int GROUP, bool CAUSAL>
__global__ void __launch_bounds__(256) row_attn_kernel(const RowAttnArgs a, unsigned int *status) {
    constexpr int E = D / 32;
    constexpr int CH = 4;  // keys per step
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
    const int t = (int)(gw / a.hkv), g = (int)(gw % a.hkv);
    if (t >= a.total) return;
    const int hq = a.hkv * GROUP;

    // segment of row t: last s with cu[s] <= t
    int lo = 0, hi = a.n_seg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int s0 = a.cu[lo], s1 = a.cu[lo + 1];
    if (!(0 <= s0 && s0 <= t && t < s1 && s1 <= a.total) || a.cu[a.n_seg] != a.total) {
        if (lane == 0) atomicOr(status, QA_DEVICE_BAD_SEGMENTS);
        return;
    }
    const int kend = CAUSAL ? t + 1 : s1;

    float q[GROUP][E], acc[GROUP][E], m[GROUP], l[GROUP];
#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
        load_bf16<E>(a.q + ((size_t)t * hq + g * GROUP + i) * D + lane * E, q[i]);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            q[i][e] *= a.scale_log2;
            acc[i][e] = 0.f;
        }
        m[i] = -INFINITY;
        l[i] = 0.f;
    }

    for (int j = s0; j < kend; j += CH) {
        const int n = min(CH, kend - j);
        float sc[GROUP][CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            if (c < n) {
                float kx[E];
                load_bf16<E>(a.k + ((size_t)(j + c) * a.hkv + g) * D + lane * E, kx);
#pragma unroll
                for (int i = 0; i < GROUP; ++i) {
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) d += q[i][e] * kx[e];
                    sc[i][c] = d;
                }
            } else {
#pragma unroll
                for (int i = 0; i < GROUP; ++i) sc[i][c] = -INFINITY;
            }
        }
#pragma unroll
        for (int i = 0; i < GROUP; ++i)
#pragma unroll
            for (int c = 0; c < CH; ++c)
                if (c < n) sc[i][c] = warp_sum(sc[i][c]);
#pragma unroll
        for (int i = 0; i < GROUP; ++i) {
            float mx = m[i];
#pragma unroll
            for (int c = 0; c < CH; ++c) mx = fmaxf(mx, sc[i][c]);
            const float alpha = exp2_approx(m[i] - mx);
            m[i] = mx;
            l[i] *= alpha;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[i][e] *= alpha;
        }
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            if (c < n) {
                float vx[E];
                load_bf16<E>(a.v + ((size_t)(j + c) * a.hkv + g) * D + lane * E, vx);
#pragma unroll
                for (int i = 0; i < GROUP; ++i) {
                    const float p = exp2_approx(sc[i][c] - m[i]);
                    l[i] += p;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[i][e] += p * vx[e];
                }
            }
        }
    }

#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
        const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
        float o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = acc[i][e] * inv;
        store_bf16<E>(a.out + ((size_t)t * hq + g * GROUP + i) * D + lane * E, o);
    }
}

}  // namespace qa
