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
// because both ranges are ordered), then counts itself in the arrival counter
// of (request, KV head); the warp that arrives last merges every partial of
// its two query heads, writes the output and resets the counter to zero, so
// nothing ever waits on another CTA and the workspace is left as it was
// found.  Only a CTA's first and last segment can be shared with a
// neighbour; their partials stay in registers until the CTA's last page and
// are written, counted in and merged then: a release and an atomic in the
// middle of the stream had stalled the consumer warps while the memory
// system was saturated (the ring filled and the producer stopped), and
// CTAs with two segments ended ~3 us after the others.  The q rows of the
// next segment are loaded one segment ahead for the same reason.
//
// Inside a CTA.  One producer warp streams whole pages (K page and V page,
// 16 tokens x Hkv heads x 128 dims of bf16 each, contiguous in the pool) into
// a ring of shared-memory stages with the bulk-copy engine; the K page and the
// V page of a stage complete on separate mbarriers, so scores start while V
// is still in flight.  The producer's lanes fetch the page ids 32 at a time.
// Hkv consumer warps share every stage: warp g handles KV head g of the page
// (all 16 tokens) and both query heads of that KV head (GQA sharing).  Lane l owns dims [4l, 4l + 4): it forms partial dot products for
// the 32 (token, head) pairs with packed fp32 FMAs, a butterfly
// reduce-scatter over the warp leaves pair l's full score on lane l, so each
// lane runs one exponential of the fp32 online softmax, and the probabilities
// reach every lane through 256 bytes of shared memory for the P V update.
// Every consumer waits on every stage it reads, in order, so no mbarrier
// phase is ever skipped.
#include <cuda_runtime.h>
#include <math.h>
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

struct DecodeArgs {
    const uint16_t *q;
    const uint8_t *k_pages;
    const uint8_t *v_pages;
    const int32_t *page_table;
    const int32_t *seq_lens;
    uint16_t *out;
    float *part_acc;  // [slots][Hq][D]
    float *part_ml;   // [slots][Hq][2]
    int *arrivals;    // [kDecodeMaxBatch][kMaxHkv], zero between calls
    int batch, hkv, max_pages, num_pages;
    float scale_log2;  // scale * log2(e)
    // lengths and page table may be read before the preceding kernel ends
    // (qa_attn_params::stable_metadata >= 1), and the pools too (>= 2)
    int early, early_pools;
    // fused decode step only: q is the pre-norm projection; the new token's
    // pre-norm k and its v are appended at position seq_lens[b] - 1
    const uint16_t *k_new, *v_new;  // [B][Hkv][D]
    const float *q_gain, *k_gain;   // [D]
    uint8_t *k_pages_w, *v_pages_w; // the pools, written at the new token's slot
    float eps;
    // theta^(-2i/D), computed on the host in fp64, as fp32 hi + lo parts
    float freq_hi[kD / 2], freq_lo[kD / 2];
};

// Per-head QK-norm and NEOX RoPE of one head vector spread over a warp
// (qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder": RMSNorm over
// head_dim with a [head_dim] gain, then rotate-half RoPE).  Lane l holds dims
// [4l, 4l + 4) in x01/x23; dim d pairs with d +- 64, which lives on lane
// l ^ 16.  gn: the gain of the lane's four dims; cs/sn: cos/sin of the
// angles of the lane's four pairs.  Returns
// the rotated dims rounded to bf16 (the operator boundary), as two packed
// words.  Warp-collective.
__device__ __forceinline__ uint2 norm_rope4(float2 x01, float2 x23, float4 gn, float eps, const float *cs,
                                            const float *sn, int lane) {
    const float ss = warp_sum(x01.x * x01.x + x01.y * x01.y + x23.x * x23.x + x23.y * x23.y);
    const float r = 1.0f / sqrtf(ss * (1.0f / kD) + eps);
    const float y[4] = {x01.x * r * gn.x, x01.y * r * gn.y, x23.x * r * gn.z, x23.y * r * gn.w};
    float z[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float p = __shfl_xor_sync(0xffffffffu, y[c], 16);  // the pair's other element
        z[c] = lane < 16 ? y[c] * cs[c] - p * sn[c] : p * sn[c] + y[c] * cs[c];
    }
    return make_uint2(pack_bf16x2(z[0], z[1]), pack_bf16x2(z[2], z[3]));
}

// cos/sin of the angles pos * theta^(-2i/D) of pairs i = 4 (l mod 16) + c
// (positions below 2^18; the host rejects longer page tables).
__device__ __forceinline__ void rope_angles(const DecodeArgs &a, int pos, int lane, float *cs, float *sn) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int i = 4 * (lane & 15) + c;
        sincos_pos_freq(pos, a.freq_hi[i], a.freq_lo[i], &sn[c], &cs[c]);
    }
}

// Pages request b contributes; invalid lengths contribute none (and are
// reported once by CTA 0).
template <bool APPEND>
__device__ __forceinline__ int pages_of(const DecodeArgs &a, int b, bool report) {
    int L = a.seq_lens[b];
    if (L < (APPEND ? 1 : 0) || L > a.max_pages * kPS) {
        if (report) atomicOr(&g_status, QA_DEVICE_BAD_LENGTH);
        return 0;
    }
    return (L + kPS - 1) / kPS;
}

struct SmemLayout {
    uint32_t stage_bytes;  // one stage: K page + V page
    uint32_t page_bytes;
    uint32_t off_bar, off_flag, off_prefix, off_pbuf, total;
};

__host__ __device__ inline SmemLayout smem_layout(int hkv, int batch, int group) {
    SmemLayout s;
    s.page_bytes = kPS * hkv * kD * 2;
    s.stage_bytes = 2 * s.page_bytes;
    uint32_t o = kStages * s.stage_bytes;
    s.off_bar = o;  // full_k[kStages], full_v[kStages], empty[kStages]
    o += 3 * kStages * 8;
    s.off_flag = o;  // page_ok[kStages]
    o += kStages * 4;
    o = (o + 15) & ~15u;
    s.off_prefix = o;
    o += (batch + 1) * 4;
    o = (o + 15) & ~15u;
    s.off_pbuf = o;  // 32 float2 per consumer warp
    o += hkv * 32 * 8;
    s.total = o;
    return s;
}

// Workspace: the arrival counters first, in a region of fixed size (one int
// per request and KV head up to the largest batch), so they sit at the same place whatever
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
    w.acc = ((size_t)kDecodeMaxBatch * kMaxHkv * sizeof(int) + 255) & ~(size_t)255;
    w.ml = w.acc + ((slots * hq * kD * sizeof(float) + 255) & ~(size_t)255);
    w.total = w.ml + ((slots * hq * 2 * sizeof(float) + 255) & ~(size_t)255);
    return w;
}

// First request b whose pages reach past page index x (prefix[b + 1] > x).
__device__ __forceinline__ int first_request_past(const int *prefix, int batch, int x) {
    int l = 0, r = batch - 1;
    while (l < r) {
        const int mid = (l + r) >> 1;
        if (prefix[mid + 1] > x) r = mid; else l = mid + 1;
    }
    return l;
}

__device__ __forceinline__ int atom_add_relaxed_gpu(int *p, int v) {
    int old;
    asm volatile("atom.add.relaxed.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void bf16x4(uint2 w, float2 &lo, float2 &hi) {
    lo = make_float2(bf16lo(w.x), bf16hi(w.x));
    hi = make_float2(bf16lo(w.y), bf16hi(w.y));
}

template <int GROUP, bool APPEND>
__global__ void __launch_bounds__((kMaxHkv + 1) * 32, 1) decode_splitk_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = smem_layout(a.hkv, a.batch, GROUP);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_consumers = a.hkv;
    const int hq = a.hkv * GROUP;

    int *prefix = reinterpret_cast<int *>(smem + L.off_prefix);
    int *page_ok = reinterpret_cast<int *>(smem + L.off_flag);  // page id of each stage, -1 if invalid
    const uint32_t bar_full_k = smem_u32(smem + L.off_bar);
    const uint32_t bar_full_v = bar_full_k + kStages * 8;
    const uint32_t bar_empty = bar_full_v + kStages * 8;

    // Launched as a programmatic dependent: wait for the previous kernel on the
    // stream to finish (and its writes to land) before touching global
    // memory -- or, when the caller vouches that lengths and page table are
    // not its output (a.early), only before touching anything else -- and
    // then let the next one start its own prologue early.  The trigger comes
    // after the wait in both modes, so a kernel that starts early on this
    // one's trigger never overlaps a kernel older than this one.
    if (!a.early) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }

    // Prefix sums of page counts over requests (warp 0), barrier init.
    if (warp == 0) {
        int carry = 0;
        if (lane == 0) prefix[0] = 0;
        for (int base = 0; base < a.batch; base += 32) {
            int b = base + lane;
            int v = b < a.batch ? pages_of<APPEND>(a, b, blockIdx.x == 0) : 0;
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
                mbar_init(bar_full_k + 8 * s, 1);
                mbar_init(bar_full_v + 8 * s, 1);
                mbar_init(bar_empty + 8 * s, n_consumers);
            }
            fence_mbar_init();
        }
    }
    __syncthreads();

    const int total = prefix[a.batch];
    const int per = (total + gridDim.x - 1) / gridDim.x;
    const int lo = blockIdx.x * per;
    const int hi = min(lo + per, total);
    // Requests b0 (holding page lo) .. b_last (holding page hi - 1).  Visit
    // order: b_last, then b0 .. b_last - 1 (see the header comment).
    const int b0 = lo < hi ? first_request_past(prefix, a.batch, lo) : 0;
    const int b_last = lo < hi ? first_request_past(prefix, a.batch, hi - 1) : -1;
    const int n_visit = lo < hi ? b_last - b0 + 1 : 0;
    // the producer's first 32 page ids (page table only)
    int first_ids = -1;
    if (warp == n_consumers && n_visit > 0) {
        const int p0 = prefix[b_last];
        const int j0 = max(lo, p0) - p0, j1 = min(hi, prefix[b_last + 1]) - p0;
        first_ids = j0 + lane < j1 ? a.page_table[(size_t)b_last * a.max_pages + j0 + lane] : -1;
    }
    // Fused step: the rotation angles of the first request visited (they
    // depend on its length only) are computed before the wait when lengths
    // may be read early.
    float cs_first[4], sn_first[4];
    const bool angles_first = APPEND && a.early && warp < n_consumers && n_visit > 0;
    if (angles_first) rope_angles(a, a.seq_lens[b_last] - 1, lane, cs_first, sn_first);
    // With the pools vouched for too (a.early_pools) the producer warp starts
    // streaming its first kStages pages before it waits (below).
    const bool producer_first = a.early_pools && warp == n_consumers;
    if (a.early && !producer_first) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }

    // CTA 0 writes the zero rows of requests with nothing to attend over
    // (threads that have waited only).
    if (blockIdx.x == 0) {
        const int chunks = hq * kD * 2 / 16;  // 16-byte chunks per request
        const int n_thr = producer_first ? n_consumers * 32 : (int)blockDim.x;
        for (int b = 0; b < a.batch && (int)threadIdx.x < n_thr; ++b) {
            if (prefix[b + 1] != prefix[b]) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + (size_t)b * hq * kD);
            for (int c = threadIdx.x; c < chunks; c += n_thr) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
    }

    if (total == 0 || lo >= hi) {
        if (producer_first) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        }
        return;
    }

    // Warm L2 with the per-request rows read at the start of every later
    // segment (q; for the fused step the new token's k and v too), so those
    // segments do not start with a round trip to HBM.
    if (warp < n_consumers) {
        for (int k = 1 + lane; k < n_visit; k += 32) {
            const int b = b0 + k - 1;
            const uint8_t *qrow = reinterpret_cast<const uint8_t *>(a.q + ((size_t)b * hq + warp * GROUP) * kD);
#pragma unroll
            for (int o = 0; o < GROUP * kD * 2; o += 128) prefetch_l2(qrow + o);
            if (APPEND) {
                const size_t o = ((size_t)b * a.hkv + warp) * kD;
                prefetch_l2(a.k_new + o);
                prefetch_l2(a.k_new + o + 64);
                prefetch_l2(a.v_new + o);
                prefetch_l2(a.v_new + o + 64);
            }
        }
    }

    if (warp == n_consumers) {
        // ---------------- producer warp: lanes fetch page ids, lane 0 issues copies
        const uint64_t policy = policy_evict_first();
        int it = 0;
        bool waited = !producer_first;
        for (int k = 0; k < n_visit; ++k) {
            const int b = k == 0 ? b_last : b0 + k - 1;
            const int p0 = prefix[b], p1 = prefix[b + 1];
            if (p1 == p0) continue;
            const int j0 = max(lo, p0) - p0, j1 = min(hi, p1) - p0;
            const int32_t *row = a.page_table + (size_t)b * a.max_pages;
            for (int jb = j0; jb < j1; jb += 32) {
                const int mine = (k == 0 && jb == j0) ? first_ids : (jb + lane < j1 ? row[jb + lane] : -1);
                const int cnt = min(32, j1 - jb);
                for (int u = 0; u < cnt; ++u, ++it) {
                    const int page = __shfl_sync(0xffffffffu, mine, u);
                    if (!waited && it == kStages) {  // the ring is full: wait now (warp-uniform)
                        asm volatile("griddepcontrol.wait;" ::: "memory");
                        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
                        waited = true;
                    }
                    if (lane == 0) {
                        const int s = it % kStages;
                        if (it >= kStages) mbar_wait(bar_empty + 8 * s, ((it / kStages) & 1) ^ 1, &g_status);
                        uint8_t *dst = smem + s * L.stage_bytes;
                        if (page < 0 || page >= a.num_pages) {
                            atomicOr(&g_status, QA_DEVICE_BAD_PAGE);
                            page_ok[s] = -1;
                            mbar_arrive(bar_full_k + 8 * s);
                            mbar_arrive(bar_full_v + 8 * s);
                        } else {
                            page_ok[s] = page;
                            const size_t off = (size_t)page * L.page_bytes;
                            mbar_arrive_expect_tx(bar_full_k + 8 * s, L.page_bytes);
                            bulk_g2s_hint(smem_u32(dst), a.k_pages + off, L.page_bytes, bar_full_k + 8 * s, policy);
                            mbar_arrive_expect_tx(bar_full_v + 8 * s, L.page_bytes);
                            bulk_g2s_hint(smem_u32(dst + L.page_bytes), a.v_pages + off, L.page_bytes,
                                          bar_full_v + 8 * s, policy);
                        }
                    }
                    __syncwarp();
                }
            }
        }
        if (!waited) {  // fewer than kStages pages
            asm volatile("griddepcontrol.wait;" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        }
        return;
    }

    // ---------------- consumer warps: warp g takes KV head g of every page
    const int g = warp;
    float2 *pbuf = reinterpret_cast<float2 *>(smem + L.off_pbuf) + warp * 32;
    // After the reduce-scatter lane l holds the score of (token my_t, query
    // head my_h of the group); with GROUP == 1 lanes l and l ^ 1 agree.
    constexpr int NV = 16 * GROUP;  // (token, head) pairs per page
    constexpr int LOG = GROUP == 2 ? 5 : 4;
    const int my_t = lane >> 1;
    const int my_h = GROUP == 2 ? lane & 1 : 0;
    const bool p_writer = GROUP == 2 ? true : (lane & 1) == 0;
    int it = 0;
    // The q rows of the next segment are loaded one segment ahead, so a
    // segment does not start with a round trip to memory.
    auto load_q = [&](int b, uint2 (&w)[GROUP]) {
#pragma unroll
        for (int i = 0; i < GROUP; ++i)
            w[i] = *reinterpret_cast<const uint2 *>(a.q + ((size_t)b * hq + g * GROUP + i) * kD + 4 * lane);
    };
    uint2 q_next[GROUP];
    load_q(b_last, q_next);
    // Partials of split segments (at most two per CTA: the first and the
    // last request of its range; the ones between are whole) are kept in
    // registers and written, counted in and merged after the last page, so
    // no segment switch waits on a release or an atomic while pages stream.
    int n_def = 0, def_b[2] = {0, 0};
    float def_acc[2][GROUP][4], def_m[2][GROUP], def_l[2][GROUP];
    for (int k = 0; k < n_visit; ++k) {
        const int b = k == 0 ? b_last : b0 + k - 1;
        uint2 qw[GROUP];
#pragma unroll
        for (int i = 0; i < GROUP; ++i) qw[i] = q_next[i];
        if (k + 1 < n_visit) load_q(b0 + k, q_next);  // segment k + 1 is request b0 + k
        const int p0 = prefix[b], p1 = prefix[b + 1];
        if (p1 == p0) continue;
        const int j0 = max(lo, p0) - p0, j1 = min(hi, p1) - p0;
        const int seq_len = a.seq_lens[b];

        float2 q01[GROUP], q23[GROUP], acc01[GROUP], acc23[GROUP];
        // fused step: the new token's K/V rows for KV head g (rotated k,
        // bf16) when this segment holds the request's last page
        const bool has_new = APPEND && j1 == p1 - p0;
        uint2 k_new_w = make_uint2(0u, 0u), v_new_w = make_uint2(0u, 0u);
        float4 gain_q = make_float4(0.f, 0.f, 0.f, 0.f), gain_k = gain_q;
        if (APPEND) {
            gain_q = *reinterpret_cast<const float4 *>(a.q_gain + 4 * lane);
            if (has_new) {
                const size_t o = ((size_t)b * a.hkv + g) * kD + 4 * lane;
                k_new_w = *reinterpret_cast<const uint2 *>(a.k_new + o);
                v_new_w = *reinterpret_cast<const uint2 *>(a.v_new + o);
                gain_k = *reinterpret_cast<const float4 *>(a.k_gain + 4 * lane);
            }
        }
        float cs[4], sn[4];
        if (APPEND) {
            if (k == 0 && angles_first) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    cs[c] = cs_first[c];
                    sn[c] = sn_first[c];
                }
            } else {
                rope_angles(a, seq_len - 1, lane, cs, sn);
            }
            if (has_new) {
                float2 k01, k23;
                bf16x4(k_new_w, k01, k23);
                k_new_w = norm_rope4(k01, k23, gain_k, a.eps, cs, sn, lane);
            }
        }
#pragma unroll
        for (int i = 0; i < GROUP; ++i) {
            uint2 w = qw[i];
            if (APPEND) {
                float2 x01, x23;
                bf16x4(w, x01, x23);
                w = norm_rope4(x01, x23, gain_q, a.eps, cs, sn, lane);
            }
            bf16x4(w, q01[i], q23[i]);
            q01[i].x *= a.scale_log2;
            q01[i].y *= a.scale_log2;
            q23[i].x *= a.scale_log2;
            q23[i].y *= a.scale_log2;
            acc01[i] = make_float2(0.f, 0.f);
            acc23[i] = make_float2(0.f, 0.f);
        }
        float m_own = -INFINITY, l_own = 0.f;

        for (int j = j0; j < j1; ++j, ++it) {
            const int s = it % kStages;
            const uint32_t phase = (it / kStages) & 1;
            mbar_wait(bar_full_k + 8 * s, phase, &g_status);
            const int nt = min(kPS, seq_len - j * kPS);
            const int page = page_ok[s];
            // fused step: this page holds the new token (last slot in use)
            const bool patch = APPEND && has_new && j == j1 - 1 && page >= 0;
            if (page >= 0 && nt > 0) {
                uint8_t *Ks = smem + s * L.stage_bytes + (g * kD + 4 * lane) * 2;
                uint8_t *Vs = Ks + L.page_bytes;
                const int row_stride = a.hkv * kD * 2;
                if (patch) {
                    // the row this lane reads is its own 8 bytes: no warp sync needed
                    const size_t off = ((size_t)page * kPS + (nt - 1)) * row_stride + (g * kD + 4 * lane) * 2;
                    *reinterpret_cast<uint2 *>(Ks + (nt - 1) * row_stride) = k_new_w;
                    *reinterpret_cast<uint2 *>(a.k_pages_w + off) = k_new_w;
                    *reinterpret_cast<uint2 *>(a.v_pages_w + off) = v_new_w;
                }
                // partial dots of every (token, head); rows past the sequence
                // (sentinels, possibly NaN) only ever touch their own entry
                float v[NV];
#pragma unroll
                for (int t = 0; t < kPS; ++t) {
                    float2 k01, k23;
                    bf16x4(*reinterpret_cast<const uint2 *>(Ks + t * row_stride), k01, k23);
#pragma unroll
                    for (int i = 0; i < GROUP; ++i) {
                        const float2 sp = ffma2(q23[i], k23, ffma2(q01[i], k01, make_float2(0.f, 0.f)));
                        v[t * GROUP + i] = sp.x + sp.y;
                    }
                }
                // butterfly reduce-scatter: stage `st` halves the live entries
#pragma unroll
                for (int st = 0; st < LOG; ++st) {
                    const int off = 16 >> st;
                    const int hn = NV >> (st + 1);
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int i = 0; i < hn; ++i) {
                        const float send = upper ? v[i] : v[i + hn];
                        const float keep = upper ? v[i + hn] : v[i];
                        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
                if (GROUP == 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
                const float sc = my_t < nt ? v[0] : -INFINITY;
                // online softmax of this lane's query head (max over the 16 token lanes)
                float tmax = sc;
#pragma unroll
                for (int off = 2; off < 32; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
                const float m_new = fmaxf(m_own, tmax);
                const float alpha_own = exp2_approx(m_own - m_new);
                const float p = exp2_approx(sc - m_new);
                l_own = l_own * alpha_own + p;
                m_own = m_new;
                float alpha[GROUP];
                if (GROUP == 2) {
                    const float other = __shfl_xor_sync(0xffffffffu, alpha_own, 1);
                    alpha[0] = my_h == 0 ? alpha_own : other;
                    alpha[GROUP - 1] = my_h == 1 ? alpha_own : other;
                } else {
                    alpha[0] = alpha_own;
                }
#pragma unroll
                for (int i = 0; i < GROUP; ++i) {
                    if (alpha[i] != 1.f) {  // uniform across the warp
                        acc01[i].x *= alpha[i];
                        acc01[i].y *= alpha[i];
                        acc23[i].x *= alpha[i];
                        acc23[i].y *= alpha[i];
                    }
                }
                __syncwarp();
                if (p_writer) pbuf[GROUP == 2 ? lane : (lane >> 1)] = make_float2(p, p);
                __syncwarp();
                mbar_wait(bar_full_v + 8 * s, phase, &g_status);
                if (patch) *reinterpret_cast<uint2 *>(Vs + (nt - 1) * row_stride) = v_new_w;
                if (nt == kPS) {
#pragma unroll
                    for (int t = 0; t < kPS; ++t) {
                        float2 v01, v23;
                        bf16x4(*reinterpret_cast<const uint2 *>(Vs + t * row_stride), v01, v23);
#pragma unroll
                        for (int i = 0; i < GROUP; ++i) {
                            const float2 pp = pbuf[t * GROUP + i];
                            acc01[i] = ffma2(v01, pp, acc01[i]);
                            acc23[i] = ffma2(v23, pp, acc23[i]);
                        }
                    }
                } else {
                    for (int t = 0; t < nt; ++t) {  // tail page: skip rows past the sequence
                        float2 v01, v23;
                        bf16x4(*reinterpret_cast<const uint2 *>(Vs + t * row_stride), v01, v23);
#pragma unroll
                        for (int i = 0; i < GROUP; ++i) {
                            const float2 pp = pbuf[t * GROUP + i];
                            acc01[i] = ffma2(v01, pp, acc01[i]);
                            acc23[i] = ffma2(v23, pp, acc23[i]);
                        }
                    }
                }
            } else {
                mbar_wait(bar_full_v + 8 * s, phase, &g_status);  // the stage is reused only once V landed
            }
            // generic stores into the stage come before the next bulk copy into it
            if (patch) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }

        // Sum of probabilities per query head over its 16 token lanes (bit 0
        // of the lane is the head, or a duplicate when GROUP == 1), and both
        // heads' (m, l) on every lane.
        float l_head = l_own;
#pragma unroll
        for (int off = 2; off < 32; off <<= 1) l_head += __shfl_xor_sync(0xffffffffu, l_head, off);
        float m[GROUP], l[GROUP], acc[GROUP][4];
        if (GROUP == 2) {
            const float m_other = __shfl_xor_sync(0xffffffffu, m_own, 1);
            const float l_other = __shfl_xor_sync(0xffffffffu, l_head, 1);
            m[0] = my_h == 0 ? m_own : m_other;
            l[0] = my_h == 0 ? l_head : l_other;
            m[GROUP - 1] = my_h == 1 ? m_own : m_other;
            l[GROUP - 1] = my_h == 1 ? l_head : l_other;
        } else {
            m[0] = m_own;
            l[0] = l_head;
        }
#pragma unroll
        for (int i = 0; i < GROUP; ++i) {
            acc[i][0] = acc01[i].x;
            acc[i][1] = acc01[i].y;
            acc[i][2] = acc23[i].x;
            acc[i][3] = acc23[i].y;
        }

        const bool whole = (j0 == 0 && j1 == p1 - p0);
        if (whole) {
#pragma unroll
            for (int i = 0; i < GROUP; ++i) {
                const int h = g * GROUP + i;
                const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
                uint2 w;
                w.x = pack_bf16x2(acc[i][0] * inv, acc[i][1] * inv);
                w.y = pack_bf16x2(acc[i][2] * inv, acc[i][3] * inv);
                *reinterpret_cast<uint2 *>(a.out + ((size_t)b * hq + h) * kD + 4 * lane) = w;
            }
        } else {
            // warp-uniform; a third split segment cannot occur (see above)
#pragma unroll
            for (int d = 0; d < 2; ++d) {
                if (d != n_def) continue;
                def_b[d] = b;
#pragma unroll
                for (int i = 0; i < GROUP; ++i) {
                    def_m[d][i] = m[i];
                    def_l[d][i] = l[i];
#pragma unroll
                    for (int e = 0; e < 4; ++e) def_acc[d][i][e] = acc[i][e];
                }
            }
            n_def = min(n_def + 1, 2);
        }
    }

    // The split segments' partials: written to slot c + b, counted in the
    // arrival counter of (request, KV head); the last arriving warp merges.
#pragma unroll
    for (int d = 0; d < 2; ++d) {
        if (d >= n_def) continue;
        const int slot = blockIdx.x + def_b[d];
#pragma unroll
        for (int i = 0; i < GROUP; ++i) {
            const int h = g * GROUP + i;
            *reinterpret_cast<float4 *>(a.part_acc + ((size_t)slot * hq + h) * kD + 4 * lane) =
                make_float4(def_acc[d][i][0], def_acc[d][i][1], def_acc[d][i][2], def_acc[d][i][3]);
            if (lane == 0) {
                a.part_ml[((size_t)slot * hq + h) * 2 + 0] = def_m[d][i];
                a.part_ml[((size_t)slot * hq + h) * 2 + 1] = def_l[d][i];
            }
        }
    }
    // the warp barrier orders every lane's partials before lane 0's
    // release fence; both arrivals then leave together, and lane 0's
    // acquire fence orders the reads of the merges after them
    __syncwarp();
    int prev[2] = {0, 0};
    if (lane == 0 && n_def > 0) {
        fence_acq_rel_gpu();
#pragma unroll
        for (int d = 0; d < 2; ++d)
            if (d < n_def) prev[d] = atom_add_relaxed_gpu(a.arrivals + (size_t)def_b[d] * kMaxHkv + g, 1);
        fence_acq_rel_gpu();
    }
#pragma unroll
    for (int d = 0; d < 2; ++d) {
        if (d >= n_def) continue;
        const int b = def_b[d];
        const int p0 = prefix[b], p1 = prefix[b + 1];
        const int c_lo = p0 / per, c_hi = (p1 - 1) / per;
        if (__shfl_sync(0xffffffffu, prev[d], 0) != c_hi - c_lo) continue;
        // online merge over batches of up to 8 partials per query head, the
        // loads of both heads of the group all in flight together (one L2
        // round trip per batch; requests of this workload span a few CTAs)
        constexpr int kBatch = 8;
        float mm[GROUP], ls[GROUP], o[GROUP][4];
#pragma unroll
        for (int i = 0; i < GROUP; ++i) {
            mm[i] = -INFINITY;
            ls[i] = 0.f;
            o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        }
        for (int c0 = c_lo; c0 <= c_hi; c0 += kBatch) {
            float mc[GROUP][kBatch], lc[GROUP][kBatch];
            float4 pv[GROUP][kBatch];
#pragma unroll
            for (int i = 0; i < GROUP; ++i) {
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (c0 + u <= c_hi) {
                        const size_t r = (size_t)(c0 + u + b) * hq + g * GROUP + i;
                        mc[i][u] = __ldcg(a.part_ml + r * 2);
                        lc[i][u] = __ldcg(a.part_ml + r * 2 + 1);
                        pv[i][u] = __ldcg(reinterpret_cast<const float4 *>(a.part_acc + r * kD + 4 * lane));
                    } else {
                        mc[i][u] = -INFINITY;
                        lc[i][u] = 0.f;
                        pv[i][u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < GROUP; ++i) {
                float mb = mm[i];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) mb = fmaxf(mb, mc[i][u]);
                if (mb == -INFINITY) continue;  // nothing attended so far
                const float alpha = exp2_approx(mm[i] - mb);  // 0 while mm = -inf
                ls[i] *= alpha;
                o[i][0] *= alpha;
                o[i][1] *= alpha;
                o[i][2] *= alpha;
                o[i][3] *= alpha;
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const float w = exp2_approx(mc[i][u] - mb);  // 0 for an empty partial (mc = -inf)
                    ls[i] += w * lc[i][u];
                    o[i][0] += w * pv[i][u].x;
                    o[i][1] += w * pv[i][u].y;
                    o[i][2] += w * pv[i][u].z;
                    o[i][3] += w * pv[i][u].w;
                }
                mm[i] = mb;
            }
        }
#pragma unroll
        for (int i = 0; i < GROUP; ++i) {
            const int h = g * GROUP + i;
            const float inv = ls[i] > 0.f ? 1.f / ls[i] : 0.f;
            uint2 w;
            w.x = pack_bf16x2(o[i][0] * inv, o[i][1] * inv);
            w.y = pack_bf16x2(o[i][2] * inv, o[i][3] * inv);
            *reinterpret_cast<uint2 *>(a.out + ((size_t)b * hq + h) * kD + 4 * lane) = w;
        }
        if (lane == 0) a.arrivals[(size_t)b * kMaxHkv + g] = 0;  // ready for the next call
    }
}

// One CTA waits on a barrier that nothing ever completes: the bounded wait
// the kernels use must give up after limit_ns, set QA_DEVICE_TIMEOUT in this
// file's status word and let the kernel end (qa_check_bounded_wait).
__global__ void bounded_wait_check_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(b, 0, &g_status, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_wait_check(unsigned int limit_us, cudaStream_t stream) {
    bounded_wait_check_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_us * 1000ull);
    return cudaGetLastError();
}

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
                          const qa_attn_params &p, float scale, int ctas, cudaStream_t stream,
                          const DecodeAppend *app) {
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
    a.early = (p.abi_version >= 2 && p.stable_metadata >= 1) ? 1 : 0;
    a.early_pools = (p.abi_version >= 2 && p.stable_metadata >= 2) ? 1 : 0;
    a.k_new = a.v_new = nullptr;
    a.q_gain = a.k_gain = nullptr;
    a.k_pages_w = a.v_pages_w = nullptr;
    a.eps = 0.f;
    for (int i = 0; i < kD / 2; ++i) a.freq_hi[i] = a.freq_lo[i] = 0.f;
    if (app) {
        a.k_new = static_cast<const uint16_t *>(app->k_new);
        a.v_new = static_cast<const uint16_t *>(app->v_new);
        a.q_gain = app->q_gain;
        a.k_gain = app->k_gain;
        a.k_pages_w = static_cast<uint8_t *>(app->k_pages);
        a.v_pages_w = static_cast<uint8_t *>(app->v_pages);
        a.eps = app->rms_eps;
        for (int i = 0; i < kD / 2; ++i) {
            const double f = pow((double)app->rope_theta, -2.0 * i / kD);
            a.freq_hi[i] = (float)f;
            a.freq_lo[i] = (float)(f - (double)a.freq_hi[i]);
        }
    }

    const SmemLayout L = smem_layout(a.hkv, batch, group);
    // programmatic dependent launch: the kernel's prologue overlaps the tail of
    // the previous kernel on the stream (it waits before touching memory)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3((a.hkv + 1) * 32);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kernel = app ? (group == 2 ? decode_splitk_kernel<2, true> : decode_splitk_kernel<1, true>)
                      : (group == 2 ? decode_splitk_kernel<2, false> : decode_splitk_kernel<1, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return e;
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
