// Tensor-core flash attention over packed segments (tcgen05 + TMEM + TMA),
// persistent and warp-specialised.
//
// A job is one 128-row query tile of one query head h of one segment (a
// prefill request or an encoder window) together with its key tiles: every
// key tile of the segment (window, bidirectional) or key tiles 0..qt (causal
// prefill, query tile qt).  A persistent grid of one CTA per SM walks the jobs
// in a fixed order; six warps share the work:
//
//   warp 4 (producer)   TMA loads: the Q tile once per job into a Q buffer,
//                       then K and V tiles ([128 rows][D] bf16, 128B-swizzled,
//                       64-dim sub-tiles) into a ring of stages.
//   warp 5 (MMA)        one thread issues S = Q K^T (M = 128, N = 128 keys,
//                       K = D in steps of 16) into one of two TMEM score
//                       buffers, one step ahead of O += P_hi V + P_lo V
//                       (M = 128, N = 64 per MMA, K = 128 keys in steps of 16,
//                       V read MN-major) into one of two TMEM output buffers;
//                       completions are signalled with tcgen05.commit.
//   warps 0-3 (softmax) thread r owns query row r (= TMEM lane r): it reads its
//                       scores with tcgen05.ld, masks keys outside the segment
//                       (and, causal, keys after the row), runs the online
//                       softmax in fp32 with base-2 exponentials, writes P as
//                       two bf16 terms P_hi = bf16(p), P_lo = bf16(p - P_hi)
//                       (128B-swizzled K-major tiles; P_lo goes into the key
//                       tile's shared memory, dead once S is computed), and
//                       rescales its row of O in TMEM when the running max
//                       moves.  At the end of a job it reads O back, divides by
//                       the softmax sum, rounds to bf16 and stores the row.
//
// The P_hi + P_lo pair carries p to about 16 significant bits, so the P V
// product keeps the softmax probabilities at (nearly) fp32 precision, as the
// precision policy asks (score and softmax intermediates in float32).
//
// Masks.  Window: key j is visible to row i iff both lie in the segment.
// Causal prefill: additionally j <= i.  Rows past the segment end are computed
// on whatever the tile holds and never stored; keys past it get probability 0,
// and their V rows (the next segment's, or TMA's zero fill past the tensor)
// are finite, so they contribute exactly 0.
//
// Every wait is bounded (common.cuh): a wait that expires sets
// QA_DEVICE_TIMEOUT and the kernel runs on to its end instead of hanging.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "tc.cuh"

namespace qa {

struct AttnTcArgs {
    const int32_t *cu;  // [n_seg + 1]
    uint16_t *out;      // [T][hq][D]
    int n_seg, total, hq;
    int qtiles;         // causal: query tiles per segment in the job list
    int n_items;        // causal: n_seg * qtiles * hq; window: n_seg * hq
    float scale_log2;
};

template <int D>
struct AttnTcLayout {
    static constexpr int kSub = D / 64;        // 64-dim sub-tiles per row block
    static constexpr int NQ = D == 64 ? 2 : 1;  // Q buffers
    static constexpr int NS = D == 64 ? 3 : 2;  // K/V stages
    static constexpr uint32_t kQBytes = kSub * tc::kSubTileBytes;
    static constexpr uint32_t kKRegion = (kSub > 2 ? kSub : 2) * tc::kSubTileBytes;  // K tile, then P_lo
    static constexpr uint32_t kVBytes = kSub * tc::kSubTileBytes;
    static constexpr uint32_t kStageBytes = kKRegion + kVBytes;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffStage = kOffQ + NQ * kQBytes;
    static constexpr uint32_t kOffP = kOffStage + NS * kStageBytes;  // P_hi: 128 keys = 2 sub-tiles
    static constexpr uint32_t kOffBar = kOffP + 2 * tc::kSubTileBytes;
    // mbarriers: q_full[NQ], q_empty[NQ], kv_full[NS], kv_empty[NS], s_full[2],
    // s_empty[2], p_full, p_empty, o_full[2], o_empty[2]
    static constexpr int kNumBars = 2 * NQ + 2 * NS + 4 + 2 + 4;
    static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr uint32_t kBytes = kOffTmemSlot + 16;
    static constexpr uint32_t kSmem = kBytes + 1024;  // slack for 1024-byte alignment
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;    // S buffers at columns 0 and 128
    static constexpr uint32_t kColO = 256;  // O buffers at columns 256 and 256 + D
};

// The job list, walked identically by every role of a CTA.
struct JobWalker {
    const AttnTcArgs &a;
    int item, qt, qt_end;
    int h, seg, s0, s1, n_tiles;

    __device__ explicit JobWalker(const AttnTcArgs &args) : a(args), item(-1), qt(0), qt_end(0) {}

    // Advances to the next job; false when the CTA has none left.  Segments
    // whose offsets are malformed are skipped (and reported when `report`).
    template <bool CAUSAL>
    __device__ bool next(unsigned int *status, bool report) {
        while (true) {
            if (qt + 1 < qt_end) {
                ++qt;
                return true;
            }
            item = item < 0 ? (int)blockIdx.x : item + (int)gridDim.x;
            if (item >= a.n_items) return false;
            int qtb = 0;
            h = item % a.hq;
            if (CAUSAL) {
                const int rest = item / a.hq;
                qtb = rest % a.qtiles;
                seg = rest / a.qtiles;
            } else {
                seg = item / a.hq;
            }
            s0 = a.cu[seg];
            s1 = a.cu[seg + 1];
            qt = qt_end = 0;
            if (!(0 <= s0 && s0 <= s1 && s1 <= a.total) || a.cu[a.n_seg] != a.total) {
                if (report) atomicOr(status, QA_DEVICE_BAD_SEGMENTS);
                continue;
            }
            n_tiles = (s1 - s0 + 127) / 128;
            if (CAUSAL) {
                if (qtb >= n_tiles) continue;
                qt = qtb;
                qt_end = qtb + 1;
            } else {
                if (n_tiles == 0) continue;
                qt_end = n_tiles;
            }
            return true;
        }
    }
    template <bool CAUSAL>
    __device__ int key_tiles() const {
        return CAUSAL ? qt + 1 : n_tiles;
    }
    __device__ int q0() const { return s0 + qt * 128; }
};

template <int D, int GROUP, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnTcArgs a, unsigned int *status) {
    using L = AttnTcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const uint32_t q_full = sb + L::kOffBar, q_empty = q_full + 8 * L::NQ;
    const uint32_t kv_full = q_empty + 8 * L::NQ, kv_empty = kv_full + 8 * L::NS;
    const uint32_t s_full = kv_empty + 8 * L::NS, s_empty = s_full + 16;
    const uint32_t p_full = s_empty + 16, p_empty = p_full + 8;
    const uint32_t o_full = p_empty + 8, o_empty = o_full + 16;

    if (tid == 0) {
        for (int i = 0; i < L::NQ; ++i) {
            mbar_init(q_full + 8 * i, 1);
            mbar_init(q_empty + 8 * i, 1);
        }
        for (int i = 0; i < L::NS; ++i) {
            mbar_init(kv_full + 8 * i, 1);
            mbar_init(kv_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + 8 * i, 1);
            mbar_init(s_empty + 8 * i, 4);
            mbar_init(o_full + 8 * i, 1);
            mbar_init(o_empty + 8 * i, 4);
        }
        mbar_init(p_full, 4);
        mbar_init(p_empty, 1);
        fence_mbar_init();
    }
    if (warp == 5) tc::tmem_alloc(sb + L::kOffTmemSlot, L::kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kOffTmemSlot);

    if (warp == 4) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            tc::prefetch_tmap(&tm_q);
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            JobWalker jw(a);
            int qi = 0, si = 0;
            while (jw.next<CAUSAL>(status, false)) {
                const int g = jw.h / GROUP;
                const int qb = qi % L::NQ;
                if (qi >= L::NQ) mbar_wait(q_empty + 8 * qb, ((qi / L::NQ) & 1) ^ 1, status);
                mbar_arrive_expect_tx(q_full + 8 * qb, L::kQBytes);
#pragma unroll
                for (int sd = 0; sd < L::kSub; ++sd)
                    tc::tma_load_3d(sb + L::kOffQ + qb * L::kQBytes + sd * tc::kSubTileBytes, &tm_q, sd * 64, jw.h,
                                    jw.q0(), q_full + 8 * qb);
                ++qi;
                const int n_kt = jw.key_tiles<CAUSAL>();
                for (int kt = 0; kt < n_kt; ++kt, ++si) {
                    const int st = si % L::NS;
                    if (si >= L::NS) mbar_wait(kv_empty + 8 * st, ((si / L::NS) & 1) ^ 1, status);
                    const uint32_t base = sb + L::kOffStage + st * L::kStageBytes;
                    mbar_arrive_expect_tx(kv_full + 8 * st, 2 * L::kSub * tc::kSubTileBytes);
                    const int k0 = jw.s0 + kt * 128;
#pragma unroll
                    for (int sd = 0; sd < L::kSub; ++sd) {
                        tc::tma_load_3d(base + sd * tc::kSubTileBytes, &tm_k, sd * 64, g, k0, kv_full + 8 * st);
                        tc::tma_load_3d(base + L::kKRegion + sd * tc::kSubTileBytes, &tm_v, sd * 64, g, k0,
                                        kv_full + 8 * st);
                    }
                }
            }
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16(128, 128, false);
            constexpr uint32_t idesc_o = tc::idesc_bf16(128, 64, true);
            JobWalker jw(a);
            int qi = 0, si = 0, sc = 0, pc = 0, job = 0;
            // the P V step still waiting for its probabilities (issued one S late)
            bool pending = false;
            int pend_st = 0, pend_job = 0, pend_kt = 0;
            bool pend_last = false;
            auto issue_pv = [&]() {
                const int obuf = pend_job & 1;
                mbar_wait(p_full, pc & 1, status);
                if (pend_kt == 0 && pend_job >= 2) mbar_wait(o_empty + 8 * obuf, ((pend_job / 2) & 1) ^ 1, status);
                tc::fence_after();
                const uint32_t stage = sb + L::kOffStage + pend_st * L::kStageBytes;
                const uint32_t o_col = tmem + L::kColO + obuf * D;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t a_off = (kk >> 2) * tc::kSubTileBytes + (kk & 3) * 32;
#pragma unroll
                    for (int sd = 0; sd < L::kSub; ++sd) {
                        const uint64_t vdesc =
                            tc::sw128_desc(stage + L::kKRegion + sd * tc::kSubTileBytes + kk * 2048);
                        tc::mma_bf16(o_col + sd * 64, tc::sw128_desc(sb + L::kOffP + a_off), vdesc, idesc_o,
                                     (pend_kt > 0 || kk > 0) ? 1u : 0u);
                        tc::mma_bf16(o_col + sd * 64, tc::sw128_desc(stage + a_off), vdesc, idesc_o, 1u);
                    }
                }
                tc::mma_commit(kv_empty + 8 * pend_st);  // K region (P_lo) and V read
                tc::mma_commit(p_empty);                  // P_hi read, O updated
                if (pend_last) tc::mma_commit(o_full + 8 * obuf);
                ++pc;
            };
            while (jw.next<CAUSAL>(status, false)) {
                const int qb = qi % L::NQ;
                const int n_kt = jw.key_tiles<CAUSAL>();
                for (int kt = 0; kt < n_kt; ++kt, ++si, ++sc) {
                    const int st = si % L::NS;
                    const int sbuf = sc & 1;
                    if (sc >= 2) mbar_wait(s_empty + 8 * sbuf, ((sc / 2) & 1) ^ 1, status);
                    if (kt == 0) mbar_wait(q_full + 8 * qb, (qi / L::NQ) & 1, status);
                    mbar_wait(kv_full + 8 * st, (si / L::NS) & 1, status);
                    tc::fence_after();
                    const uint32_t qbase = sb + L::kOffQ + qb * L::kQBytes;
                    const uint32_t kbase = sb + L::kOffStage + st * L::kStageBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * tc::kSubTileBytes + (kk & 3) * 32;
                        tc::mma_bf16(tmem + L::kColS + sbuf * 128, tc::sw128_desc(qbase + off),
                                     tc::sw128_desc(kbase + off), idesc_s, kk > 0);
                    }
                    tc::mma_commit(s_full + 8 * sbuf);
                    if (kt == n_kt - 1) tc::mma_commit(q_empty + 8 * qb);
                    if (pending) issue_pv();
                    pending = true;
                    pend_st = st;
                    pend_job = job;
                    pend_kt = kt;
                    pend_last = kt == n_kt - 1;
                }
                ++qi;
                ++job;
            }
            if (pending) issue_pv();
        }
    } else {
        // ---------------------------------------------------------- softmax / epilogue
        const int r = tid;  // query row in the tile = TMEM lane
        const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
        const uint32_t sw = (uint32_t)(r & 7);
        JobWalker jw(a);
        int si = 0, sc = 0, job = 0;
        while (jw.next<CAUSAL>(status, tid == 0)) {
            const int q0 = jw.q0(), qi = q0 + r, s1 = jw.s1;
            const int n_kt = jw.key_tiles<CAUSAL>();
            const int obuf = job & 1;
            const uint32_t o_col = tmem + t_lane + L::kColO + obuf * D;
            float m = -INFINITY, l = 0.f;
            for (int kt = 0; kt < n_kt; ++kt, ++si, ++sc) {
                const int k0 = jw.s0 + kt * 128;
                const int sbuf = sc & 1;
                const uint32_t s_col = tmem + t_lane + L::kColS + sbuf * 128;
                mbar_wait(s_full + 8 * sbuf, (sc / 2) & 1, status);
                tc::fence_after();
                const bool full_tile = (k0 + 128 <= s1) && (!CAUSAL || k0 + 127 <= q0);
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float sv[32];
                    tc::tmem_ld32(s_col + c * 32, sv);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int key = k0 + c * 32 + j;
                        const bool ok = full_tile || (key < s1 && (!CAUSAL || key <= qi));
                        if (ok) mx = fmaxf(mx, sv[j]);
                    }
                }
                const float m_new = fmaxf(m, mx * a.scale_log2);
                const float alpha = m == -INFINITY ? 0.f : exp2_approx(m - m_new);
                // P_hi is free, and O holds every earlier key tile, once the
                // previous P V step (step sc - 1 of this CTA) has completed
                if (sc > 0) mbar_wait(p_empty, (sc - 1) & 1, status);
                tc::fence_after();
                const uint32_t p_row = sb + L::kOffP + r * 128;
                const uint32_t plo_row = sb + L::kOffStage + (si % L::NS) * L::kStageBytes + r * 128;
                float psum = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float sv[32];
                    tc::tmem_ld32(s_col + c * 32, sv);
                    uint32_t pk[16], pl[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int key = k0 + c * 32 + j;
                        const bool ok0 = full_tile || (key < s1 && (!CAUSAL || key <= qi));
                        const bool ok1 = full_tile || (key + 1 < s1 && (!CAUSAL || key + 1 <= qi));
                        const float p0 = ok0 ? exp2_approx(sv[j] * a.scale_log2 - m_new) : 0.f;
                        const float p1 = ok1 ? exp2_approx(sv[j + 1] * a.scale_log2 - m_new) : 0.f;
                        psum += p0 + p1;
                        const uint32_t hi = pack_bf16x2(p0, p1);
                        pk[j >> 1] = hi;
                        pl[j >> 1] = pack_bf16x2(p0 - bf16lo(hi), p1 - bf16hi(hi));
                    }
                    // 32 keys = 4 chunks of 16 bytes, sub-tile c / 2, chunks (c % 2) * 4 + u
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t chunk = (uint32_t)((c & 1) * 4 + u);
                        const uint32_t off = (uint32_t)(c >> 1) * tc::kSubTileBytes + ((chunk ^ sw) << 4);
                        tc::st_shared_v4(p_row + off, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                        tc::st_shared_v4(plo_row + off, pl[4 * u], pl[4 * u + 1], pl[4 * u + 2], pl[4 * u + 3]);
                    }
                }
                l = l * alpha + psum;
                m = m_new;
                // rescale this row of the output accumulator (warp-collective)
                if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float ov[32];
                        tc::tmem_ld32(o_col + c * 32, ov);
#pragma unroll
                        for (int j = 0; j < 32; ++j) ov[j] *= alpha;
                        tc::tmem_st32(o_col + c * 32, ov);
                    }
                }
                tc::fence_proxy_async_smem();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(p_full);
                    mbar_arrive(s_empty + 8 * sbuf);
                }
            }
            // epilogue: O / l -> bf16 (warp-collective TMEM reads, masked stores)
            mbar_wait(o_full + 8 * obuf, (job / 2) & 1, status);
            tc::fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)qi * a.hq + jw.h) * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float ov[32];
                tc::tmem_ld32(o_col + c * 32, ov);
                if (qi < s1) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint4 w;
                        w.x = pack_bf16x2(ov[8 * u + 0] * inv, ov[8 * u + 1] * inv);
                        w.y = pack_bf16x2(ov[8 * u + 2] * inv, ov[8 * u + 3] * inv);
                        w.z = pack_bf16x2(ov[8 * u + 4] * inv, ov[8 * u + 5] * inv);
                        w.w = pack_bf16x2(ov[8 * u + 6] * inv, ov[8 * u + 7] * inv);
                        dst[c * 4 + u] = w;
                    }
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_empty + 8 * obuf);
            ++job;
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 5) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace qa
