// Paged GQA decode: split-K flash decode over a paged KV pool, with the
// split-combine folded into the same kernel.
//
// What it computes (qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder":
// decode attends over [0, cur_len + 1) of the cache; "GGUF layout": 16 query
// heads over 8 KV heads, head_dim 128; M* "Speech recognition: Whisper and
// Qwen3-ASR", "Graph": decode runs on paged KV):
//   out[b][h] = softmax_j(q[b][h] . K_b[j] * scale) V_b[j],  j < seq_lens[b],
// with K_b[j] the row of page page_table[b][j / 16], slot j % 16, KV head
// h / group.
//
// Work split.  The pages of all requests form one flat list (request-major).
// A persistent grid of one CTA per SM cuts that list into equal contiguous
// ranges, so every CTA streams the same number of pages whatever the mix of
// lengths.  A CTA's range intersects one or more requests; each intersection
// is a "segment".  A segment that holds a whole request writes the final
// bf16 output.  Otherwise it writes an fp32 partial (running max, running
// sum, un-normalised accumulator) to slot c + b (CTA c, request b: unique
// because both ranges are ordered), then counts itself in the request's
// arrival counter; the CTA that arrives last merges every partial of the
// request, writes the output and resets the counter to zero, so nothing ever
// waits on another CTA and the workspace is left as it was found.
//
// Inside a CTA.  One producer warp streams whole pages (K page and V page,
// 16 tokens x Hkv heads x 128 dims of bf16 each, contiguous in the pool) into
// a ring of shared-memory stages with the bulk-copy engine, completing on an
// mbarrier per stage; its lanes fetch the page ids 32 at a time.  2*Hkv
// consumer warps share each stage: warp (g, half) handles KV head g for tokens
// [8*half, 8*half + 8) of the page and both query heads of that KV head (GQA
// sharing), with the fp32 online softmax in registers and warp-shuffle
// reductions.  Lane l owns dims [4l, 4l + 4).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "qa_internal.h"

namespace qa {
namespace {

__device__ unsigned int g_status;

constexpr int kD = 128;
constexpr int kPS = 16;
constexpr int kStages = 3;
constexpr int kMaxHkv = 8;
// Merge record of one query head in shared memory: m, l, two pad words (so
// the accumulator starts on a 16-byte boundary), then acc[kD].
constexpr int kRec = 4 + kD;
// Named barrier over every consumer warp (ids 1..8 are the KV-head pairs).
constexpr int kBarConsumers = 9;

struct DecodeArgs {
    const uint16_t *q;
    const uint8_t *k_pages;
    const uint8_t *v_pages;
    const int32_t *page_table;
    const int32_t *seq_lens;
    uint16_t *out;
    float *part_acc;  // [slots][Hq][D]
    float *part_ml;   // [slots][Hq][2]
    int *arrivals;    // [batch], zero between calls
    int batch, hkv, max_pages, num_pages;
    float scale_log2;  // scale * log2(e)
};

// Pages request b contributes; invalid lengths contribute none (and are
// reported once by CTA 0).
__device__ __forceinline__ int pages_of(const DecodeArgs &a, int b, bool report) {
    int L = a.seq_lens[b];
    if (L < 0 || L > a.max_pages * kPS) {
        if (report) atomicOr(&g_status, QA_DEVICE_BAD_LENGTH);
        return 0;
    }
    return (L + kPS - 1) / kPS;
}

struct SmemLayout {
    uint32_t stage_bytes;  // one stage: K page + V page
    uint32_t page_bytes;
    uint32_t off_bar, off_flag, off_prefix, off_merge, total;
};

__host__ __device__ inline SmemLayout smem_layout(int hkv, int batch, int group) {
    SmemLayout s;
    s.page_bytes = kPS * hkv * kD * 2;
    s.stage_bytes = 2 * s.page_bytes;
    uint32_t o = kStages * s.stage_bytes;
    s.off_bar = o;
    o += 2 * kStages * 8;
    s.off_flag = o;  // page_ok[kStages], then the "merge here" flag
    o += (kStages + 1) * 4;
    o = (o + 15) & ~15u;
    s.off_prefix = o;
    o += (batch + 1) * 4;
    o = (o + 15) & ~15u;
    s.off_merge = o;
    o += hkv * group * kRec * 4;
    s.total = o;
    return s;
}

// Workspace: the arrival counters first, in a region of fixed size (one int
// per request up to the largest batch), so they sit at the same place whatever
// the batch of a call; then the partials, whose placement depends on the
// batch.  A zero-filled workspace therefore stays valid across calls of
// different batch sizes: each call only touches counters it leaves at zero.
struct WorkspaceLayout {
    size_t arrivals, acc, ml, total;
};

__host__ __device__ inline WorkspaceLayout workspace_layout(int batch, int hq, int ctas) {
    const size_t slots = (size_t)ctas + (size_t)batch;
    WorkspaceLayout w;
    w.arrivals = 0;
    w.acc = ((size_t)kDecodeMaxBatch * sizeof(int) + 255) & ~(size_t)255;
    w.ml = w.acc + ((slots * hq * kD * sizeof(float) + 255) & ~(size_t)255);
    w.total = w.ml + ((slots * hq * 2 * sizeof(float) + 255) & ~(size_t)255);
    return w;
}

template <int GROUP>
__global__ void __launch_bounds__((2 * kMaxHkv + 1) * 32, 1) decode_splitk_kernel(const DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = smem_layout(a.hkv, a.batch, GROUP);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_consumers = 2 * a.hkv;
    const int hq = a.hkv * GROUP;

    int *prefix = reinterpret_cast<int *>(smem + L.off_prefix);
    int *page_ok = reinterpret_cast<int *>(smem + L.off_flag);
    volatile int *merge_here = reinterpret_cast<volatile int *>(smem + L.off_flag) + kStages;
    const uint32_t bar_full = smem_u32(smem + L.off_bar);
    const uint32_t bar_empty = bar_full + kStages * 8;

    // Prefix sums of page counts over requests (warp 0), barrier init.
    if (warp == 0) {
        int carry = 0;
        if (lane == 0) prefix[0] = 0;
        for (int base = 0; base < a.batch; base += 32) {
            int b = base + lane;
            int v = b < a.batch ? pages_of(a, b, blockIdx.x == 0) : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (b < a.batch) prefix[b + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(bar_full + 8 * s, 1);
                mbar_init(bar_empty + 8 * s, n_consumers);
            }
            fence_mbar_init();
        }
    }
    __syncthreads();

    // CTA 0 writes the zero rows of requests with nothing to attend over.
    if (blockIdx.x == 0) {
        const int chunks = hq * kD * 2 / 16;  // 16-byte chunks per request
        for (int b = 0; b < a.batch; ++b) {
            if (prefix[b + 1] != prefix[b]) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + (size_t)b * hq * kD);
            for (int c = threadIdx.x; c < chunks; c += blockDim.x) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
    }

    const int total = prefix[a.batch];
    if (total == 0) return;
    const int per = (total + gridDim.x - 1) / gridDim.x;
    const int lo = blockIdx.x * per;
    const int hi = min(lo + per, total);
    if (lo >= hi) return;

    // First request whose pages reach past lo.
    int b0 = 0;
    {
        int l = 0, r = a.batch - 1;
        while (l < r) {
            int mid = (l + r) >> 1;
            if (prefix[mid + 1] > lo) r = mid; else l = mid + 1;
        }
        b0 = l;
    }

    if (warp == n_consumers) {
        // ---------------- producer warp: lanes fetch page ids, lane 0 issues copies
        const uint64_t policy = policy_evict_first();
        int it = 0;
        for (int b = b0; b < a.batch && prefix[b] < hi; ++b) {
            const int p0 = prefix[b], p1 = prefix[b + 1];
            if (p1 == p0) continue;
            const int j0 = max(lo, p0) - p0, j1 = min(hi, p1) - p0;
            const int32_t *row = a.page_table + (size_t)b * a.max_pages;
            for (int jb = j0; jb < j1; jb += 32) {
                const int mine = jb + lane < j1 ? row[jb + lane] : -1;
                const int cnt = min(32, j1 - jb);
                for (int u = 0; u < cnt; ++u, ++it) {
                    const int page = __shfl_sync(0xffffffffu, mine, u);
                    if (lane == 0) {
                        const int s = it % kStages;
                        if (it >= kStages) mbar_wait(bar_empty + 8 * s, ((it / kStages) & 1) ^ 1, &g_status);
                        uint8_t *dst = smem + s * L.stage_bytes;
                        if (page < 0 || page >= a.num_pages) {
                            atomicOr(&g_status, QA_DEVICE_BAD_PAGE);
                            page_ok[s] = 0;
                            mbar_arrive(bar_full + 8 * s);
                        } else {
                            page_ok[s] = 1;
                            mbar_arrive_expect_tx(bar_full + 8 * s, L.stage_bytes);
                            const size_t off = (size_t)page * L.page_bytes;
                            bulk_g2s_hint(smem_u32(dst), a.k_pages + off, L.page_bytes, bar_full + 8 * s, policy);
                            bulk_g2s_hint(smem_u32(dst + L.page_bytes), a.v_pages + off, L.page_bytes,
                                          bar_full + 8 * s, policy);
                        }
                    }
                    __syncwarp();
                }
            }
        }
        return;
    }

    // ---------------- consumer warps
    const int g = warp >> 1, half = warp & 1;
    float *merge = reinterpret_cast<float *>(smem + L.off_merge) + g * GROUP * kRec;
    int it = 0;
    for (int b = b0; b < a.batch && prefix[b] < hi; ++b) {
        const int p0 = prefix[b], p1 = prefix[b + 1];
        if (p1 == p0) continue;
        const int j0 = max(lo, p0) - p0, j1 = min(hi, p1) - p0;
        const int seq_len = a.seq_lens[b];

        float q[GROUP][4], acc[GROUP][4], m[GROUP], l[GROUP];
#pragma unroll
        for (int i = 0; i < GROUP; ++i) {
            const uint2 w = *reinterpret_cast<const uint2 *>(
                a.q + ((size_t)b * hq + g * GROUP + i) * kD + 4 * lane);
            q[i][0] = bf16lo(w.x) * a.scale_log2;
            q[i][1] = bf16hi(w.x) * a.scale_log2;
            q[i][2] = bf16lo(w.y) * a.scale_log2;
            q[i][3] = bf16hi(w.y) * a.scale_log2;
            m[i] = -INFINITY;
            l[i] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
        }

        for (int j = j0; j < j1; ++j, ++it) {
            const int s = it % kStages;
            mbar_wait(bar_full + 8 * s, (it / kStages) & 1, &g_status);
            const int n_valid = min(kPS, seq_len - j * kPS);
            const int t0 = half * 8;
            const int nt = min(8, n_valid - t0);
            if (page_ok[s] && nt > 0) {
                const uint8_t *Ks = smem + s * L.stage_bytes;
                const uint8_t *Vs = Ks + L.page_bytes;
                float sc[GROUP][8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (t < nt) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(
                            Ks + (((t0 + t) * a.hkv + g) * kD + 4 * lane) * 2);
                        const float k0 = bf16lo(w.x), k1 = bf16hi(w.x), k2 = bf16lo(w.y), k3 = bf16hi(w.y);
#pragma unroll
                        for (int i = 0; i < GROUP; ++i)
                            sc[i][t] = warp_sum(q[i][0] * k0 + q[i][1] * k1 + q[i][2] * k2 + q[i][3] * k3);
                    } else {
#pragma unroll
                        for (int i = 0; i < GROUP; ++i) sc[i][t] = -INFINITY;
                    }
                }
#pragma unroll
                for (int i = 0; i < GROUP; ++i) {
                    float mx = m[i];
#pragma unroll
                    for (int t = 0; t < 8; ++t) mx = fmaxf(mx, sc[i][t]);
                    const float alpha = exp2_approx(m[i] - mx);
                    m[i] = mx;
                    l[i] *= alpha;
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[i][e] *= alpha;
                }
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (t < nt) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(
                            Vs + (((t0 + t) * a.hkv + g) * kD + 4 * lane) * 2);
                        const float v0 = bf16lo(w.x), v1 = bf16hi(w.x), v2 = bf16lo(w.y), v3 = bf16hi(w.y);
#pragma unroll
                        for (int i = 0; i < GROUP; ++i) {
                            const float p = exp2_approx(sc[i][t] - m[i]);
                            l[i] += p;
                            acc[i][0] += p * v0;
                            acc[i][1] += p * v1;
                            acc[i][2] += p * v2;
                            acc[i][3] += p * v3;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }

        // Merge the two halves of KV head g through shared memory.
        if (half == 1) {
#pragma unroll
            for (int i = 0; i < GROUP; ++i) {
                float *mr = merge + i * kRec;
                if (lane == 0) {
                    mr[0] = m[i];
                    mr[1] = l[i];
                }
                *reinterpret_cast<float4 *>(mr + 4 + 4 * lane) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            }
        }
        named_barrier(1 + g, 64);
        const bool whole = (j0 == 0 && j1 == p1 - p0);
        if (half == 0) {
            const int slot = blockIdx.x + b;
#pragma unroll
            for (int i = 0; i < GROUP; ++i) {
                const float *mr = merge + i * kRec;
                const float m1 = mr[0], l1 = mr[1];
                const float4 a1 = *reinterpret_cast<const float4 *>(mr + 4 + 4 * lane);
                const float mm = fmaxf(m[i], m1);
                float ls = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
                if (mm != -INFINITY) {
                    const float c0 = exp2_approx(m[i] - mm), c1 = exp2_approx(m1 - mm);
                    ls = l[i] * c0 + l1 * c1;
                    o[0] = acc[i][0] * c0 + a1.x * c1;
                    o[1] = acc[i][1] * c0 + a1.y * c1;
                    o[2] = acc[i][2] * c0 + a1.z * c1;
                    o[3] = acc[i][3] * c0 + a1.w * c1;
                }
                const int h = g * GROUP + i;
                if (whole) {
                    const float inv = ls > 0.f ? 1.f / ls : 0.f;
                    uint2 w;
                    w.x = pack_bf16x2(o[0] * inv, o[1] * inv);
                    w.y = pack_bf16x2(o[2] * inv, o[3] * inv);
                    *reinterpret_cast<uint2 *>(a.out + ((size_t)b * hq + h) * kD + 4 * lane) = w;
                } else {
                    *reinterpret_cast<float4 *>(a.part_acc + ((size_t)slot * hq + h) * kD + 4 * lane) =
                        make_float4(o[0], o[1], o[2], o[3]);
                    if (lane == 0) {
                        a.part_ml[((size_t)slot * hq + h) * 2 + 0] = mm;
                        a.part_ml[((size_t)slot * hq + h) * 2 + 1] = ls;
                    }
                    __threadfence();  // the partial is visible device-wide before the arrival below
                }
            }
        }
        named_barrier(1 + g, 64);

        if (!whole) {
            // Count this segment in; the last of the request's segments merges.
            const int c_lo = p0 / per, c_hi = (p1 - 1) / per;
            named_barrier(kBarConsumers, n_consumers * 32);
            if (threadIdx.x == 0) {
                const int prev = atomicAdd(a.arrivals + b, 1);
                *merge_here = (prev == c_hi - c_lo);
            }
            named_barrier(kBarConsumers, n_consumers * 32);
            if (*merge_here) {
                __threadfence();
                for (int h = warp; h < hq; h += n_consumers) {
                    float mm = -INFINITY, ls = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int c = c_lo; c <= c_hi; ++c) {
                        const size_t r = (size_t)(c + b) * hq + h;
                        const float mc = __ldcg(a.part_ml + r * 2), lc = __ldcg(a.part_ml + r * 2 + 1);
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part_acc + r * kD + 4 * lane));
                        const float mn = fmaxf(mm, mc);
                        if (mn == -INFINITY) continue;
                        const float so = exp2_approx(mm - mn), sn = exp2_approx(mc - mn);
                        ls = ls * so + lc * sn;
                        o[0] = o[0] * so + v.x * sn;
                        o[1] = o[1] * so + v.y * sn;
                        o[2] = o[2] * so + v.z * sn;
                        o[3] = o[3] * so + v.w * sn;
                        mm = mn;
                    }
                    const float inv = ls > 0.f ? 1.f / ls : 0.f;
                    uint2 w;
                    w.x = pack_bf16x2(o[0] * inv, o[1] * inv);
                    w.y = pack_bf16x2(o[2] * inv, o[3] * inv);
                    *reinterpret_cast<uint2 *>(a.out + ((size_t)b * hq + h) * kD + 4 * lane) = w;
                }
                if (threadIdx.x == 0) a.arrivals[b] = 0;  // ready for the next call
            }
        }
    }
}

}  // namespace

int decode_grid_ctas(int device) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
        return 0;
    return sms;
}

size_t decode_workspace_bytes(int batch, int n_q_heads, int head_dim, int ctas) {
    (void)head_dim;
    return workspace_layout(batch, n_q_heads, ctas).total;
}

cudaError_t launch_decode(const void *q, const void *k_pages, const void *v_pages,
                          const int32_t *page_table, const int32_t *seq_lens, int batch, void *out,
                          const qa_attn_params &p, float scale, int ctas, cudaStream_t stream) {
    const int group = p.n_q_heads / p.n_kv_heads;
    const WorkspaceLayout W = workspace_layout(batch, p.n_q_heads, ctas);
    uint8_t *ws = static_cast<uint8_t *>(p.workspace);
    DecodeArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k_pages = static_cast<const uint8_t *>(k_pages);
    a.v_pages = static_cast<const uint8_t *>(v_pages);
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.out = static_cast<uint16_t *>(out);
    a.part_acc = reinterpret_cast<float *>(ws + W.acc);
    a.part_ml = reinterpret_cast<float *>(ws + W.ml);
    a.arrivals = reinterpret_cast<int *>(ws + W.arrivals);
    a.batch = batch;
    a.hkv = p.n_kv_heads;
    a.max_pages = p.max_pages_per_seq;
    a.num_pages = p.num_pages;
    a.scale_log2 = scale * kLog2e;

    const SmemLayout L = smem_layout(a.hkv, batch, group);
    const int threads = (2 * a.hkv + 1) * 32;
    cudaError_t e;
    if (group == 2) {
        e = cudaFuncSetAttribute(decode_splitk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
        if (e != cudaSuccess) return e;
        decode_splitk_kernel<2><<<ctas, threads, L.total, stream>>>(a);
    } else {
        e = cudaFuncSetAttribute(decode_splitk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
        if (e != cudaSuccess) return e;
        decode_splitk_kernel<1><<<ctas, threads, L.total, stream>>>(a);
    }
    return cudaGetLastError();
}

unsigned int status_read_clear_decode(cudaStream_t stream, cudaError_t *err) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && v) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (err) *err = e;
    return v;
}

}  // namespace qa
