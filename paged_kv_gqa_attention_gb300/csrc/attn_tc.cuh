// Tensor-core flash attention over packed segments (tcgen05 + TMEM + TMA):
// the AuT window attention (window_tc_kernel) and the causal prefill with
// its KV page write (prefill_tc_kernel).  A job is the 128-row query tiles
// of one query head of one segment (an encoder window, or one query tile of
// a prefill request); CTAs have four warps.  The window kernel is persistent
// (small, uniform jobs: barriers and TMEM set up once per CTA, the next
// job's tiles requested while the current one finishes); the prefill runs
// one CTA per job (uneven jobs, balanced by the hardware scheduler).  Per key
// tile of 128 rows:
//   1. TMA brings the K and V tiles ([128 rows][D] bf16, 128B-swizzled, 64-dim
//      sub-tiles) and the Q tile into shared memory; Q + K and V complete on
//      separate mbarriers, so S starts before V is in.
//   2. One thread issues S = Q K^T (M = 128, N = 128 keys, K = D in steps of
//      16) into TMEM columns [0, 128) and commits to an mbarrier.
//   3. Thread r owns query row r (= TMEM lane r): it reads its scores with
//      tcgen05.ld, keeps the first n_ok keys of the tile (the rest lie outside
//      the segment or, causal, after the row), runs the online softmax in fp32
//      with base-2 exponentials, and writes P as two bf16 terms, P_hi = p
//      truncated to bf16 and P_lo = bf16(p - P_hi) (softmax_tile: P_hi in
//      TMEM over the consumed scores; P_lo in the dead Q/K shared memory for
//      the window kernel, in TMEM too for the prefill).  The pair carries p to
//      about 16 significant bits, so the P V product keeps the softmax
//      probabilities at (nearly) fp32 precision, as the precision policy asks
//      (score and softmax intermediates in float32).
//   4. The reference max m of a row (exponentials are taken relative to it)
//      moves only when a tile's max exceeds it by more than kRescaleSlack
//      (8, in log2 units): below that the probabilities stay <= 2^8 and the
//      row keeps m, so O and the sum need no rescaling (softmax is invariant
//      under the choice of reference; the sum uses the same one).  When it
//      moves, the thread rescales its row of the fp32 output accumulator O
//      in TMEM by alpha = 2^(m_old - m_new).
//   5. One thread issues O += P_hi V and O += P_lo V (M = 128, N = 64 per
//      MMA, K = 128 keys in steps of 16, V read MN-major).
// After the last key tile each row of O is read back, divided by its softmax
// sum, rounded to bf16 and staged in shared memory; the window kernel writes
// the stage out with TMA stores of 32-row boxes (store_rows_tma), the prefill
// with whole rows per warp store (store_rows_staged).
//
// Masks.  Window: key j is visible to row i iff both lie in the segment.
// Causal prefill: additionally j <= i.  Rows past the segment end are computed
// on whatever the tile holds and never stored; keys past it get probability 0,
// and their V rows (the next segment's, or TMA's zero fill past the tensor)
// are finite, so they contribute exactly 0.
//
// Every wait is bounded (common.cuh): one that expires sets QA_DEVICE_TIMEOUT
// and the kernel runs on to its end instead of hanging.
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
    float scale_log2;
    // causal prefill: the KV page write (k_pages == nullptr: none)
    const int32_t *page_table;     // [n_seg][max_pages]
    uint16_t *k_pages, *v_pages;   // [num_pages][page_size][hkv][D]
    int hkv, max_pages, num_pages, page_size;
    // chunked prefill: cached positions per request (nullptr: none)
    const int32_t *n_past;
    // prefill: segments, cached lengths and page table may be read before the
    // kernel before this one has finished (qa_attn_params::stable_metadata)
    int early;
    // window: job counter in caller memory (two words, zero), or nullptr for
    // the static job order
    int *job_ctr;
};

template <int D>
struct AttnTcLayout {
    static constexpr int kSub = D / 64;  // 64-dim sub-tiles per row block
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kSub * tc::kSubTileBytes;
    static constexpr uint32_t kV = kK + kSub * tc::kSubTileBytes;
    // P_lo (128 keys = 2 sub-tiles): over Q and K when D = 64 (Q is reloaded
    // with every key tile), over K when D = 128
    static constexpr uint32_t kPlo = D == 64 ? kQ : kK;
    static constexpr uint32_t kBar = kV + kSub * tc::kSubTileBytes;  // 4 mbarriers
    static constexpr uint32_t kTmemSlot = kBar + 32;
    static constexpr uint32_t kNext = kTmemSlot + 8;  // next-job records (persistent kernels; the prefill's job)
    static constexpr uint32_t kBytes = kNext + 32;
    static constexpr uint32_t kSmem = kBytes + 1024;  // slack for 1024-byte alignment
};

// Online softmax of one 128-key tile for this thread's query row, whose
// scores sit in TMEM columns [0, 128) of s_row (window kernel).  Keys
// [0, n_ok) of the tile are visible.  Writes P as P_hi (bf16, two keys per
// column) over the scores in columns [0, 64) and P_lo as a 128B-swizzled
// K-major row at plo_row (shared memory).  Two passes over the scores (max,
// then exponentials), each reading them from TMEM.  Updates the running
// (m, l) and, when `rescale` and m moved, multiplies the row of O at o_row
// by 2^(m_old - m_new).  Warp-collective (every lane of the warp calls it).
// Slack of the lazy reference max, in log2 units: probabilities stay <= 2^8.
constexpr float kRescaleSlack = 8.f;

template <int D>
__device__ __forceinline__ void softmax_tile(uint32_t s_row, int n_ok, float scale_log2, uint32_t plo_row,
                                             uint32_t sw, uint32_t o_row, bool rescale, float &m, float &l) {
    const int warp_max = __reduce_max_sync(0xffffffffu, n_ok);
    const int warp_min = __reduce_min_sync(0xffffffffu, n_ok);
    // TMEM reads are software-pipelined: chunk c + 1 (32 columns) is in
    // flight while chunk c is processed; dead chunks (warp-uniform) are
    // neither read nor computed.
    const int n_chunks = (warp_max + 31) >> 5;
    // the last live chunk holds at most 16 live keys: its upper half is
    // neither reduced nor exponentiated (its probabilities are written as 0)
    const bool half_tail = warp_max - (n_chunks - 1) * 32 <= 16;
    const uint32_t plo_sw = plo_row | (sw << 4);
    uint32_t ra[32], rb[32];
    // four independent running maxima and sums: no reduction is one long
    // dependency chain
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    tc::tmem_ld32_issue(s_row, ra);
    tc::tmem_ld32_wait(ra);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c >= n_chunks) break;
        uint32_t(&cur)[32] = (c & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (c & 1) ? ra : rb;
        if (c + 1 < n_chunks) tc::tmem_ld32_issue(s_row + (c + 1) * 32, nxt);
        // masked keys become -inf in place (only the 16 keys the max reads
        // when the chunk is a half tail)
        // and go back to TMEM, so the exponential pass reads them masked
        const bool tail_chunk = half_tail && c == n_chunks - 1;
        if (c * 32 + 32 > warp_min) {
            if (tail_chunk) {
#pragma unroll
                for (int j = 0; j < 16; ++j) cur[j] = c * 32 + j < n_ok ? cur[j] : __float_as_uint(-INFINITY);
                tc::tmem_st16(s_row + c * 32, *reinterpret_cast<const uint32_t(*)[16]>(&cur[0]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) cur[j] = c * 32 + j < n_ok ? cur[j] : __float_as_uint(-INFINITY);
                tc::tmem_st16(s_row + c * 32, *reinterpret_cast<const uint32_t(*)[16]>(&cur[0]));
                tc::tmem_st16(s_row + c * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&cur[16]));
            }
        }
#pragma unroll
        for (int j = 0; j < 16; j += 2)
            mx4[(j >> 1) & 3] = fmax3(mx4[(j >> 1) & 3], __uint_as_float(cur[j]), __uint_as_float(cur[j + 1]));
        if (!tail_chunk) {
#pragma unroll
            for (int j = 16; j < 32; j += 2)
                mx4[(j >> 1) & 3] = fmax3(mx4[(j >> 1) & 3], __uint_as_float(cur[j]), __uint_as_float(cur[j + 1]));
        }
        if (c + 1 < n_chunks) tc::tmem_ld32_wait(nxt);
    }
    const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
    // lazy reference max (step 4 of the header); the first tile (m = -inf)
    // always sets it
    const float m_new = mx > m + kRescaleSlack ? mx : m;
    const float alpha = m == -INFINITY ? 0.f : exp2_approx(m - m_new);
    float2 psum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    const float2 scale2 = make_float2(scale_log2, scale_log2);
    const float2 neg_m2 = make_float2(-m_new, -m_new);
    tc::tmem_wait_st();  // the masked chunk's write-back lands before it is read again
    tc::tmem_ld32_issue(s_row, ra);
    tc::tmem_ld32_wait(ra);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t(&cur)[32] = (c & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (c & 1) ? ra : rb;
        const bool live = c < n_chunks;  // warp-uniform: a dead chunk gets zero probabilities
        if (live && c + 1 < n_chunks) tc::tmem_ld32_issue(s_row + (c + 1) * 32, nxt);
        // the chunk's 32 keys in two halves of 16, each written out before
        // the next is computed (fewer registers live at once):
        // x = s * scale * log2(e) - m for a pair, on packed fp32; then
        // P_hi = p truncated to bf16 (exact), P_lo = bf16(p - P_hi)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t pk[8], pl[8];
            if (!live || (hf == 1 && half_tail && c == n_chunks - 1)) {
#pragma unroll
                for (int i = 0; i < 8; ++i) pk[i] = pl[i] = 0u;
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; jj += 2) {
                    const int j = hf * 16 + jj;
                    // masked keys read back as -inf (the max pass wrote them)
                    const float2 x =
                        ffma2(make_float2(__uint_as_float(cur[j]), __uint_as_float(cur[j + 1])), scale2, neg_m2);
                    const float2 pp = make_float2(exp2_approx(x.x), exp2_approx(x.y));
                    psum4[(j >> 1) & 3] = fadd2(psum4[(j >> 1) & 3], pp);
                    // P_hi of both keys in one word; the two truncated values
                    // back as floats from that word (a multiply by 2^16 for
                    // the low half, which the multiply-add pipe can take)
                    const uint32_t w = __byte_perm(__float_as_uint(pp.x), __float_as_uint(pp.y), 0x7632);
                    pk[jj >> 1] = w;
                    const float2 lo = fsub2(pp, make_float2(__uint_as_float(w * 65536u), __uint_as_float(w & 0xffff0000u)));
                    pl[jj >> 1] = pack_bf16x2(lo.x, lo.y);
                }
            }
            // P_hi: 16 keys = 8 TMEM columns [16c + 8hf, +8) (scores there are consumed)
            tc::tmem_st8(s_row + c * 16 + hf * 8, pk);
            // P_lo: 2 chunks of 16 bytes, sub-tile c / 2, chunks (c % 2) * 4 + 2 hf + u
            // (plo_row's bits 4-6 are zero: the swizzle is one XOR of a base
            // that already holds sw)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t chunk = (uint32_t)((c & 1) * 4 + hf * 2 + u);
                tc::st_shared_v4((plo_sw ^ (chunk << 4)) + (uint32_t)(c >> 1) * tc::kSubTileBytes, pl[4 * u],
                                 pl[4 * u + 1], pl[4 * u + 2], pl[4 * u + 3]);
            }
        }
        if (live && c + 1 < n_chunks) tc::tmem_ld32_wait(nxt);
    }
    tc::tmem_wait_st();
    const float2 psum2 = fadd2(fadd2(psum4[0], psum4[1]), fadd2(psum4[2], psum4[3]));
    l = l * alpha + (psum2.x + psum2.y);
    m = m_new;
    // rescale this row of the output accumulator (warp-collective)
    if (rescale && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tc::tmem_ld32(o_row + c * 32, ov);
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] *= alpha;
            tc::tmem_st32(o_row + c * 32, ov);
        }
    }
}

// Single-pass softmax with both P terms in TMEM (prefill), for kernels whose
// register budget holds a whole score row (two 128-thread CTAs per SM): the
// live 32-column chunks of the row are read from TMEM with one wait, the max
// and the exponentials work on the registers, and both P terms go back over
// the scores they replace: keys [32c, 32c + 32) give P_hi in columns
// [32c, 32c + 16) and P_lo in [32c + 16, 32c + 32).  The scores are read once
// instead of twice.  Same (m, l) update, lazy reference max and rescale as
// softmax_tile, the rescale of O done before any P is written.  Once keys
// [0, 64) of the row are in TMEM it calls mid() -- every thread of the CTA,
// at the same point -- so the caller can start P V on that half while the
// rest is exponentiated.  CTA-collective through mid().
template <int D, typename Mid>
__device__ __forceinline__ void softmax_tile_regs(uint32_t s_row, int n_ok, float scale_log2, uint32_t o_row,
                                                  bool rescale, float &m, float &l, Mid &&mid) {
    const int warp_max = __reduce_max_sync(0xffffffffu, n_ok);
    const int warp_min = __reduce_min_sync(0xffffffffu, n_ok);
    const int n_chunks = (warp_max + 31) >> 5;  // warp-uniform
    const bool half_tail = warp_max - (n_chunks - 1) * 32 <= 16;
    uint32_t sc[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        if (c < n_chunks) tc::tmem_ld32_issue(s_row + c * 32, sc[c]);
    // one wait for all loads; each call names its chunk, so no use of a
    // chunk moves above the wait
#pragma unroll
    for (int c = 0; c < 4; ++c)
        if (c < n_chunks) tc::tmem_ld32_wait(sc[c]);
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c >= n_chunks) break;
        if (c * 32 + 32 > warp_min) {  // masked keys become -inf in place
#pragma unroll
            for (int j = 0; j < 32; ++j) sc[c][j] = c * 32 + j < n_ok ? sc[c][j] : __float_as_uint(-INFINITY);
        }
        const bool upper = !(half_tail && c == n_chunks - 1);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            if (j >= 16 && !upper) break;
            mx4[(j >> 1) & 3] = fmax3(mx4[(j >> 1) & 3], __uint_as_float(sc[c][j]), __uint_as_float(sc[c][j + 1]));
        }
    }
    const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
    const float m_new = mx > m + kRescaleSlack ? mx : m;  // lazy reference max (see softmax_tile)
    const float alpha = m == -INFINITY ? 0.f : exp2_approx(m - m_new);
    float2 psum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    const float2 scale2 = make_float2(scale_log2, scale_log2);
    const float2 neg_m2 = make_float2(-m_new, -m_new);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c == 2) {
            // O is rescaled before any P of this tile is handed over (the
            // previous tile's P V has completed: this tile's S came after it)
            if (rescale && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    float ov[32];
                    tc::tmem_ld32(o_row + cc * 32, ov);
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] *= alpha;
                    tc::tmem_st32(o_row + cc * 32, ov);
                }
            }
            mid();  // keys [0, 64) of every row are in TMEM
        }
        uint32_t pk[16], pl[16];
        if (c >= n_chunks) {  // warp-uniform: a dead chunk gets zero probabilities
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pl[i] = 0u;
        } else {
            auto pair = [&](int j) {
                const float2 x =
                    ffma2(make_float2(__uint_as_float(sc[c][j]), __uint_as_float(sc[c][j + 1])), scale2, neg_m2);
                const float2 pp = make_float2(exp2_approx(x.x), exp2_approx(x.y));
                psum4[(j >> 1) & 3] = fadd2(psum4[(j >> 1) & 3], pp);
                const uint32_t b0 = __float_as_uint(pp.x), b1 = __float_as_uint(pp.y);
                pk[j >> 1] = __byte_perm(b0, b1, 0x7632);
                const float2 lo =
                    fsub2(pp, make_float2(__uint_as_float(b0 & 0xffff0000u), __uint_as_float(b1 & 0xffff0000u)));
                pl[j >> 1] = pack_bf16x2(lo.x, lo.y);
            };
#pragma unroll
            for (int j = 0; j < 16; j += 2) pair(j);
            if (half_tail && c == n_chunks - 1) {
#pragma unroll
                for (int i = 8; i < 16; ++i) pk[i] = pl[i] = 0u;
            } else {
#pragma unroll
                for (int j = 16; j < 32; j += 2) pair(j);
            }
        }
        tc::tmem_st16(s_row + c * 32, pk);
        tc::tmem_st16(s_row + c * 32 + 16, pl);
    }
    tc::tmem_wait_st();
    const float2 psum2 = fadd2(fadd2(psum4[0], psum4[1]), fadd2(psum4[2], psum4[3]));
    l = l * alpha + (psum2.x + psum2.y);
    m = m_new;
}

// Epilogue through shared memory: thread r (of the 128 threads that own the
// tile's rows) rounds its O row (divided by l)
// to bf16 and writes it to row r of a staging tile (D * 2 bytes per row,
// 16-byte chunk c of row r at chunk position c ^ (r & 7), so the writes of 8
// consecutive rows hit all banks); then each warp writes back its own 32 rows
// with D / 8 lanes per row, whole rows per store instruction.  Rows at or
// past row_end (= s1 - q0) are not stored.  Warp-collective; the staging rows
// of a warp are touched by that warp only.
template <int D>
__device__ __forceinline__ void store_rows_staged(uint32_t o_row, float l, uint32_t stage, uint16_t *out, int hq,
                                                  int h, int q0, int row_end, int r) {
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const int lane = r & 31, warp = r >> 5;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const uint32_t my_row = stage + (uint32_t)r * (D * 2);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tc::tmem_ld32(o_row + c * 32, ov);
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 o0 = fmul2(make_float2(ov[8 * u + 0], ov[8 * u + 1]), inv2);
            const float2 o1 = fmul2(make_float2(ov[8 * u + 2], ov[8 * u + 3]), inv2);
            const float2 o2 = fmul2(make_float2(ov[8 * u + 4], ov[8 * u + 5]), inv2);
            const float2 o3 = fmul2(make_float2(ov[8 * u + 6], ov[8 * u + 7]), inv2);
            const uint32_t chunk = (uint32_t)(c * 4 + u);
            const uint32_t pos = (chunk & ~7u) | ((chunk ^ (uint32_t)r) & 7u);
            tc::st_shared_v4(my_row + pos * 16, pack_bf16x2(o0.x, o0.y), pack_bf16x2(o1.x, o1.y),
                             pack_bf16x2(o2.x, o2.y), pack_bf16x2(o3.x, o3.y));
        }
    }
    __syncwarp();
    constexpr int kRowsPerStep = 32 / kChunks;  // rows one warp instruction covers
    const int c = lane % kChunks;
#pragma unroll
    for (int i = 0; i < 32 / kRowsPerStep; ++i) {
        const int rr = warp * 32 + i * kRowsPerStep + lane / kChunks;
        const uint32_t pos = ((uint32_t)c & ~7u) | (((uint32_t)c ^ (uint32_t)rr) & 7u);
        uint32_t x0, x1, x2, x3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                     : "r"(stage + (uint32_t)rr * (D * 2) + pos * 16));
        if (rr < row_end)
            *reinterpret_cast<uint4 *>(out + ((size_t)(q0 + rr) * hq + h) * D + c * 8) = make_uint4(x0, x1, x2, x3);
    }
}

// Rows per output TMA store box (the window output tensor map's box height):
// a 104-row window leaves in three boxes plus eight rows of plain stores.
constexpr int kOutBoxRows = 32;

// Epilogue through TMA stores: thread r stages its row of O (divided by l,
// bf16) sub-tile by sub-tile -- dims [64 sd, 64 sd + 64) of row r at stage +
// sd * 16 KiB + r * 128 with its 16-byte chunks XOR-swizzled by r, which is
// the layout of a 128B-swizzled TMA box of 64 dims (8-row swizzle atoms
// stacked) -- then thread store_tid writes the rows of whole kOutBoxRows-row
// boxes with TMA stores (tensor map tm_out, box {64, 1, kOutBoxRows}; tracked
// by that thread's bulk group: it waits for their reads of shared memory
// before the stage is reused) and the threads of the remaining rows
// (< kOutBoxRows) store theirs.  Rows at or past row_end are not written.  r
// is the thread's row (= threadIdx.x); CTA-collective (128 threads).
template <int D>
__device__ __forceinline__ void store_rows_tma(uint32_t o_row, float l, uint32_t stage, const CUtensorMap *tm_out,
                                               uint16_t *out, int hq, int h, int q0, int row_end, int r,
                                               int store_tid) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const uint32_t my_row = stage + (uint32_t)r * 128u;
    // my_row's bits 4-6 are zero: the chunk swizzle is one XOR of a base
    // that already holds r & 7
    const uint32_t my_row_sw = my_row | ((uint32_t)(r & 7) << 4);
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tc::tmem_ld32(o_row + c * 32, ov);
        const uint32_t sub = (uint32_t)(c >> 1) * tc::kSubTileBytes;  // 32 dims = half a sub-tile
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 o0 = fmul2(make_float2(ov[8 * u + 0], ov[8 * u + 1]), inv2);
            const float2 o1 = fmul2(make_float2(ov[8 * u + 2], ov[8 * u + 3]), inv2);
            const float2 o2 = fmul2(make_float2(ov[8 * u + 4], ov[8 * u + 5]), inv2);
            const float2 o3 = fmul2(make_float2(ov[8 * u + 6], ov[8 * u + 7]), inv2);
            const uint32_t chunk = (uint32_t)((c & 1) * 4 + u);
            tc::st_shared_v4((my_row_sw ^ (chunk << 4)) + sub, pack_bf16x2(o0.x, o0.y), pack_bf16x2(o1.x, o1.y),
                             pack_bf16x2(o2.x, o2.y), pack_bf16x2(o3.x, o3.y));
        }
    }
    tc::fence_proxy_async_smem();  // the staged rows are read by the TMA unit
    __syncthreads();
    const int n_rows = min(128, row_end);
    const int full = n_rows / kOutBoxRows * kOutBoxRows;
    if (r == store_tid && full > 0) {
        for (int i = 0; i < full; i += kOutBoxRows)
#pragma unroll
            for (int sd = 0; sd < D / 64; ++sd)
                tc::tma_store_3d(tm_out, stage + sd * tc::kSubTileBytes + (uint32_t)i * 128u, sd * 64, h, q0 + i);
        tc::bulk_commit_group();
    }
    if (r >= full && r < n_rows) {
        uint16_t *dst = out + ((size_t)(q0 + r) * hq + h) * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(my_row + (uint32_t)(c >> 3) * tc::kSubTileBytes +
                               ((((uint32_t)c & 7u) ^ (uint32_t)(r & 7)) << 4)));
            *reinterpret_cast<uint4 *>(dst + c * 8) = make_uint4(x0, x1, x2, x3);
        }
    }
}

// S = Q K^T (M = 128, N = 128 keys, K = D in steps of 16: 32 bytes inside a
// 128-byte row) into TMEM columns [0, 128) of tmem.  One thread.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tmem, uint32_t q_base, uint32_t k_base) {
    constexpr uint32_t idesc_s = tc::idesc_bf16(128, 128, false);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * tc::kSubTileBytes + (kk & 3) * 32;
        tc::mma_bf16(tmem, tc::sw128_desc(q_base + off), tc::sw128_desc(k_base + off), idesc_s, kk > 0);
    }
}

// O += P_hi V + P_lo V: K = 128 keys in steps of 16 (8 TMEM columns of P_hi;
// two 8-row groups of V = 2048 bytes), N = 64 dims per MMA (one V sub-tile
// each).  P_hi in TMEM columns [0, 64) of tmem, O at o_col.  One thread.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t o_col, uint32_t plo_base, uint32_t v_base,
                                         bool accumulate) {
    constexpr uint32_t idesc_o = tc::idesc_bf16(128, 64, true);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a_off = (kk >> 2) * tc::kSubTileBytes + (kk & 3) * 32;
#pragma unroll
        for (int sd = 0; sd < D / 64; ++sd) {
            const uint64_t vdesc = tc::sw128_desc(v_base + sd * tc::kSubTileBytes + kk * 2048);
            const uint32_t o = o_col + sd * 64;
            tc::mma_bf16_ts(o, tmem + kk * 8, vdesc, idesc_o, (accumulate || kk > 0) ? 1u : 0u);
            tc::mma_bf16(o, tc::sw128_desc(plo_base + a_off), vdesc, idesc_o, 1u);
        }
    }
}

// KV page write from the K and V tiles in shared memory (128B-swizzled 64-dim
// sub-tiles): tile row rr is new row i0 + rr of segment seg, at position
// i = past + i0 + rr of its request, and goes, bit for bit, to slot i % 16 of
// page page_table[seg][i / 16] (the page size is 16, the only one the
// library accepts), KV head g.  Rows at or past len, or positions past
// max_pages * 16, are not written; a page id outside [0, num_pages) sets
// QA_DEVICE_BAD_PAGE and skips the row.
//
// kv_tile_page_id, called well ahead by every thread of the 128 (tix = 0 ..
// 127, whole warps), reads the page ids: the tile's rows span at most 9
// pages, and lane j of every warp holds the j-th.  write_kv_pages (the same
// 128 threads) takes each row's page id from that lane with a shuffle.  Each
// row is written by D / 8 adjacent threads (16 bytes each), so one warp store
// covers whole 256-byte rows; a thread's rows are 8 apart, so its swizzled
// chunk offset is the same for all of them.  A null k_tile or v_tile skips
// that pool; tile rows before row_begin are left to the caller.
__device__ __forceinline__ int kv_tile_page_id(const AttnTcArgs &a, int seg, int i0, int len, int past, int tix) {
    const int lane = tix & 31;
    const int end = min(min(len, a.max_pages * 16 - past) - i0, 128);
    const int pos0 = past + i0;
    if (end > 0 && pos0 / 16 + lane <= (pos0 + end - 1) / 16) return a.page_table[(size_t)seg * a.max_pages + pos0 / 16 + lane];
    return -1;
}

template <int D>
__device__ __forceinline__ void write_kv_pages(const uint8_t *k_tile, const uint8_t *v_tile, const AttnTcArgs &a,
                                               int i0, int len, int past, int g, unsigned int *status, int tix,
                                               int my_page, int row_begin) {
    constexpr int kPage = 16;
    constexpr int kChunks = D / 8;              // 16-byte chunks per row
    constexpr int kRowsPerPass = 128 / kChunks;
    const int c = tix % kChunks, rr0 = tix / kChunks;
    const int end = min(min(len, a.max_pages * kPage - past) - i0, 128);
    const int pos0 = past + i0;  // position of tile row 0
    const int p_first = pos0 / kPage;
    // shared offset of this thread's chunk in row rr: rr * 128 + this
    const uint32_t chunk_off = (uint32_t)(c >> 3) * tc::kSubTileBytes + ((uint32_t)((c & 7) ^ (rr0 & 7)) << 4);
    const uint32_t k_s = k_tile ? smem_u32(k_tile) + chunk_off : 0u;
    const uint32_t v_s = v_tile ? smem_u32(v_tile) + chunk_off : 0u;
    const size_t row_elems = (size_t)a.hkv * D;  // one pool row (slot): all KV heads
    uint16_t *const k_dst = a.k_pages + (size_t)g * D + (size_t)c * 8;
    uint16_t *const v_dst = a.v_pages + (size_t)g * D + (size_t)c * 8;
#pragma unroll 4
    for (int k = 0; k < 128 / kRowsPerPass; ++k) {  // warp-uniform trip count
        const int rr = rr0 + k * kRowsPerPass;
        const int pos = pos0 + rr;
        const int page = __shfl_sync(0xffffffffu, my_page, (pos / kPage - p_first) & 31);
        if (rr < row_begin || rr >= end) continue;
        if (page < 0 || page >= a.num_pages) {
            if (c == 0) atomicOr(status, QA_DEVICE_BAD_PAGE);
            continue;
        }
        const size_t row = ((size_t)page * kPage + (size_t)(pos % kPage)) * row_elems;
        uint32_t x0, x1, x2, x3;
        if (k_tile) {
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(k_s + (uint32_t)rr * 128u));
            *reinterpret_cast<uint4 *>(k_dst + row) = make_uint4(x0, x1, x2, x3);
        }
        if (v_tile) {
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(v_s + (uint32_t)rr * 128u));
            *reinterpret_cast<uint4 *>(v_dst + row) = make_uint4(x0, x1, x2, x3);
        }
    }
}

// O += P_hi V + P_lo V with both P terms in TMEM in the chunk layout of
// softmax_tile_regs: keys [16kk, 16kk + 16) are P_hi columns
// 32 (kk / 2) + 8 (kk % 2) + [0, 8) and P_lo columns 16 further.  N = D:
// one MMA covers every dim, V read MN-major across its 64-wide sub-tiles
// (kSubTileBytes apart) -- half the instructions of one MMA per sub-tile,
// so the issuing thread, which also owns a softmax row, spends less time
// waiting for room in the tensor core's queue.  half = 0 / 1: keys [0, 64)
// / [64, 128) only (-1: all).  One thread.
template <int D>
__device__ __forceinline__ void issue_pv_tp(uint32_t tmem, uint32_t o_col, uint32_t v_base, bool accumulate,
                                            int half = -1) {
    constexpr uint32_t idesc_o = tc::idesc_bf16(128, D, true);
    const int kk0 = half < 0 ? 0 : 4 * half, kk1 = half < 0 ? 8 : kk0 + 4;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        if (kk < kk0 || kk >= kk1) continue;
        const uint32_t a_hi = tmem + (uint32_t)(kk >> 1) * 32 + (uint32_t)(kk & 1) * 8;
        const uint64_t vdesc = tc::sw128_desc_mn(v_base + kk * 2048, tc::kSubTileBytes);
        tc::mma_bf16_ts(o_col, a_hi, vdesc, idesc_o, (accumulate || kk > 0) ? 1u : 0u);
        tc::mma_bf16_ts(o_col, a_hi + 16, vdesc, idesc_o, 1u);
    }
}

// TMA loads of one key tile of a job (and of its query tile when load_q):
// Q and K complete on bar_qk, V on bar_v.  One thread.
template <int D>
__device__ __forceinline__ void issue_qk_loads(uint32_t sb, const CUtensorMap *tm_q, const CUtensorMap *tm_k, int h,
                                               int g, int q0, int k0, bool load_q, uint32_t bar_qk) {
    using L = AttnTcLayout<D>;
    mbar_arrive_expect_tx(bar_qk, (load_q ? 2 : 1) * L::kSub * tc::kSubTileBytes);
#pragma unroll
    for (int sd = 0; sd < L::kSub; ++sd) {
        if (load_q) tc::tma_load_3d(sb + L::kQ + sd * tc::kSubTileBytes, tm_q, sd * 64, h, q0, bar_qk);
        tc::tma_load_3d(sb + L::kK + sd * tc::kSubTileBytes, tm_k, sd * 64, g, k0, bar_qk);
    }
}

template <int D>
__device__ __forceinline__ void issue_v_loads(uint32_t sb, const CUtensorMap *tm_v, int g, int k0, uint32_t bar_v) {
    using L = AttnTcLayout<D>;
    mbar_arrive_expect_tx(bar_v, L::kSub * tc::kSubTileBytes);
#pragma unroll
    for (int sd = 0; sd < L::kSub; ++sd)
        tc::tma_load_3d(sb + L::kV + sd * tc::kSubTileBytes, tm_v, sd * 64, g, k0, bar_v);
}

// Window attention, persistent: a grid of a few CTAs per SM walks the jobs
// (window, head), job = window * n_heads + head.  CTA c takes job c first;
// after that either job c + i * gridDim.x (static order), or, with a job
// counter (a.job_ctr), the next unclaimed job in index order, so CTAs that
// run slower (later to start, or on a busier SM) take fewer jobs and every
// CTA finishes at about the same time.  Either way the CTAs running at any
// time hold every head of a run of neighbouring windows: the heads' 128-byte
// slices of a token's row (all heads side by side) are fetched at about the
// same time, which keeps DRAM pages open for the whole row rather than
// reopening them once per head.  Barriers and TMEM are set up once per CTA.
// Q + K and V land on separate barriers, so S starts before V is in.  The
// next job's Q and K are requested as soon as the current job's last P V
// has finished reading shared memory, so they load during the epilogue; the
// epilogue stages the output rows in the V buffer and writes whole rows per
// store (store_rows_tma: 32-row TMA stores), after which the next job's V is
// requested.  Each job is computed as described at the top of this file.
// TMEM: 128 columns when every job is a single 128-row tile and D = 64 (four
// CTAs share the 512 columns of an SM), else 256.
//
// The job counter is two words of caller memory, zero before the launch:
// [0] counts the claims past the first gridDim.x jobs, [1] the CTAs that
// have finished claiming; the last of those puts both back to zero, so the
// next launch on the stream finds them zero again.
template <int D>
__global__ void __launch_bounds__(128, D == 64 ? 4 : 2)
    window_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                     const AttnTcArgs a, unsigned int *status) {
    using L = AttnTcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int G = gridDim.x;
    const int n_jobs = a.n_seg * a.hq;
    // launched as a programmatic dependent: wait for the kernel before it
    // (and its writes) before reading anything, then let the next one be
    // scheduled as this grid's CTAs retire
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (a.cu[a.n_seg] != a.total) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(status, QA_DEVICE_BAD_SEGMENTS);
        return;
    }
    // does any job span more than one 128-row tile?  (With a job counter a
    // CTA's jobs are not known ahead: then every window is looked at.)
    int multi = 0;
    if (a.job_ctr) {
        for (int sg = tid; sg < a.n_seg; sg += 128) multi |= a.cu[sg + 1] - a.cu[sg] > 128;
    } else {
        for (long long j = blockIdx.x + (long long)tid * G; j < n_jobs; j += 128LL * G) {
            const int seg = (int)(j / a.hq);
            multi |= a.cu[seg + 1] - a.cu[seg] > 128;
        }
    }
    multi = __syncthreads_or(multi);
    const uint32_t tmem_cols = (D == 64 && !multi) ? 128u : 256u;

    const uint32_t bar_qk = sb + L::kBar, bar_s = bar_qk + 8, bar_o = bar_qk + 16, bar_v = bar_qk + 24;
    // Job records (job, head, s0, s1) in two shared slots.  Thread 32 fills
    // slot (i + 1) & 1 at the top of job i -- it knows that job's index one
    // job ahead (a claim made at the top of job i - 1, whose result has
    // arrived by then) -- and every thread reads slot i & 1 at the top of
    // job i (at least one CTA barrier lies between), so no job waits on a
    // claim or on a global read of the segment array.  Slot i & 1 is
    // rewritten only in job i + 2, after the barriers of job i + 1 that
    // follow every read of it.  job >= n_jobs ends the walk.  Job indices
    // stay below n_jobs + 2 G < 2^32.
    int *rec = reinterpret_cast<int *>(smem + L::kNext);
    auto fill = [&](int *slot, uint32_t j) {
        int v0 = n_jobs, v1 = 0, v2 = 0, v3 = 0;
        if (j < (uint32_t)n_jobs) {
            const uint32_t seg = j / (uint32_t)a.hq;
            v0 = (int)j;
            v1 = (int)(j - seg * (uint32_t)a.hq);
            v2 = a.cu[seg];
            v3 = a.cu[seg + 1];
        }
        slot[0] = v0;
        slot[1] = v1;
        slot[2] = v2;
        slot[3] = v3;
    };
    // the index of the job after job j (thread 32)
    auto next_index = [&](uint32_t j) -> uint32_t {
        if (j >= (uint32_t)n_jobs) return (uint32_t)n_jobs;  // no claims past the end
        return a.job_ctr ? (uint32_t)G + (uint32_t)atomicAdd(a.job_ctr, 1) : j + (uint32_t)G;
    };
    uint32_t ahead = 0;  // thread 32: index of the job after the one in the newest record
    if (tid == 0) {
        mbar_init(bar_qk, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }
    if (tid == 32) {
        fill(rec, blockIdx.x);
        ahead = next_index(blockIdx.x);
    }
    if (warp == 0) tc::tmem_alloc(sb + L::kTmemSlot, tmem_cols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);

    uint32_t ph_qk = 0, ph_v = 0, ph_s = 0, ph_o = 0;
    const int r = tid;
    const uint32_t plo_row = sb + L::kPlo + r * 128;
    const uint32_t sw = (uint32_t)(r & 7);
    bool prefetched = false;  // thread 0: the job's first Q/K tiles are already requested

    for (int it = 0;; ++it) {
        const int *cur = rec + (it & 1) * 4;
        const int job = cur[0], h = cur[1], s0 = cur[2], s1 = cur[3];
        if (job >= n_jobs) break;  // uniform: every thread read the same record
        int *nx = rec + ((it + 1) & 1) * 4;
        if (tid == 32) {  // off the MMA-issue path
            fill(nx, ahead);
            ahead = next_index(ahead);  // used at the top of the next job
        }
        const bool valid = 0 <= s0 && s0 <= s1 && s1 <= a.total;
        if (!valid && tid == 0) atomicOr(status, QA_DEVICE_BAD_SEGMENTS);
        const int n_tiles = valid ? (s1 - s0 + 127) / 128 : 0;
        if (n_tiles == 0) {
            __syncthreads();  // publishes the next record (uniform: every thread has the same bounds)
            continue;         // nothing was requested for an empty or invalid job
        }
        const bool o_in_s = D == 64 && n_tiles == 1;
        const uint32_t col_o = o_in_s ? 64u : 128u;
        // the thread that issues a job's output TMA stores and, once they
        // have read the stage (the V buffer), the next job's V: thread 96 for
        // a single-tile job, so thread 0 goes straight on to the next job's S;
        // thread 0 when the job has more query tiles, whose loads it issues
        // itself into the same buffer
        const int store_tid = n_tiles == 1 ? 96 : 0;

        for (int qt = 0; qt < n_tiles; ++qt) {
            const int q0 = s0 + qt * 128;
            float m = -INFINITY, l = 0.f;
            for (int kt = 0; kt < n_tiles; ++kt) {
                const int k0 = s0 + kt * 128;
                const bool last = qt == n_tiles - 1 && kt == n_tiles - 1;
                if (tid == 0) {
                    if (!(prefetched && qt == 0 && kt == 0)) {
                        issue_qk_loads<D>(sb, &tm_q, &tm_k, h, h, q0, k0, D == 64 || kt == 0, bar_qk);
                        issue_v_loads<D>(sb, &tm_v, h, k0, bar_v);
                    }
                    prefetched = false;
                    mbar_wait(bar_qk, ph_qk, status);
                    tc::fence_after();
                    issue_s<D>(tmem, sb + L::kQ, sb + L::kK);
                    tc::mma_commit(bar_s);
                }
                ph_qk ^= 1;
                // warp 0 waits for S; the other warps sleep in the CTA
                // barrier instead of re-testing the mbarrier
                if (warp == 0) mbar_wait(bar_s, ph_s, status);
                ph_s ^= 1;
                __syncthreads();
                tc::fence_after();

                int n_ok = min(128, s1 - k0);
                n_ok = max(n_ok, 0);
                softmax_tile<D>(t_row, n_ok, a.scale_log2, plo_row, sw, t_row + col_o, kt > 0, m, l);
                tc::fence_proxy_async_smem();
                tc::fence_before();
                __syncthreads();

                if (tid == 0) {
                    mbar_wait(bar_v, ph_v, status);
                    tc::fence_after();
                    issue_pv<D>(tmem, tmem + col_o, sb + L::kPlo, sb + L::kV, kt > 0);
                    tc::mma_commit(bar_o);
                }
                ph_v ^= 1;
                if (warp == 0) mbar_wait(bar_o, ph_o, status);  // the other warps sleep in the barrier
                ph_o ^= 1;
                __syncthreads();
                tc::fence_after();
                // Q/K/P buffers are free: request the next job's Q and K
                // (the record was published by the softmax barrier above)
                if (tid == 0 && last) {
                    const int nx_job = nx[0], nx_h = nx[1], nx_s0 = nx[2], nx_s1 = nx[3];
                    if (nx_job < n_jobs && 0 <= nx_s0 && nx_s0 < nx_s1 && nx_s1 <= a.total) {
                        issue_qk_loads<D>(sb, &tm_q, &tm_k, nx_h, nx_h, nx_s0, nx_s0, true, bar_qk);
                        prefetched = true;
                    }
                }
            }
            // epilogue staged in the V buffer (free since the last P V)
            store_rows_tma<D>(t_row + col_o, l, sb + L::kV, &tm_out, a.out, a.hq, h, q0, s1 - q0, tid, store_tid);
            tc::fence_before();
            __syncthreads();  // every TMEM read and staging read is done
            // the V buffer is free again once the TMA stores have read it:
            // after the last query tile, request the next job's V (its Q and
            // K went out under the same condition)
            if (tid == store_tid) {
                tc::bulk_wait_group_read_all();
                if (qt == n_tiles - 1) {
                    const int nx_job = nx[0], nx_h = nx[1], nx_s0 = nx[2], nx_s1 = nx[3];
                    if (nx_job < n_jobs && 0 <= nx_s0 && nx_s0 < nx_s1 && nx_s1 <= a.total)
                        issue_v_loads<D>(sb, &tm_v, nx_h, nx_s0, bar_v);
                }
            }
        }
    }

    // the CTA has made its last claim (its result was used above); the last
    // CTA to get here resets the counter for the next launch
    if (a.job_ctr && tid == 32) {
        __threadfence();
        if (atomicAdd(a.job_ctr + 1, 1) == G - 1) {
            atomicExch(a.job_ctr, 0);
            atomicExch(a.job_ctr + 1, 0);
        }
    }
    if (warp == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, tmem_cols);
    }
}

// ---------------------------------------------------------------------------
// Job order of the causal prefill.  A job (request r, query tile t) costs
// n_ct(r) + t + 1 key tiles (n_ct: cached key tiles of the chunked form, 0
// otherwise); request r has jobs at the costs lo_r = n_ct(r) + 1 .. hi_r =
// n_ct(r) + qtiles(r).  Job index jj counts the jobs in decreasing cost,
// requests in index order within a cost, so the longest jobs launch first and
// no CTA of the grid's front is spent on an empty (request, tile) slot.
// Warp-collective: reads the segment array (and the cached lengths), finds
// the cost level by a binary search over count(c) = #jobs of cost >= c, and
// the request inside the level by ballots.  Returns the request (tile in *t)
// or -1 when jj is past the last job.  Invalid segments or cached lengths
// count as empty here; the kernel checks its own request again.
__device__ __forceinline__ int prefill_job(const AttnTcArgs &a, bool past_mode, int jj, int qtiles_grid, int max_len,
                                           int *t) {
    const int lane = threadIdx.x & 31;
    auto range = [&](int r, int &lo, int &hi) {
        lo = 1;
        hi = 0;
        if (r >= a.n_seg) return;
        const int s0 = a.cu[r], s1 = a.cu[r + 1];
        const int len = (0 <= s0 && s0 <= s1 && s1 <= a.total) ? s1 - s0 : 0;
        int pst = past_mode ? a.n_past[r] : 0;
        if (pst < 0 || pst > max_len) pst = 0;
        lo = (pst + 127) / 128 + 1;
        hi = lo - 1 + min((len + 127) / 128, qtiles_grid);
    };
    int lo0, hi0;  // the first 32 requests stay in registers
    range(lane, lo0, hi0);
    auto count = [&](int c) {  // jobs of cost >= c
        int n = max(0, hi0 - max(lo0, c) + 1);
        for (int r0 = 32; r0 < a.n_seg; r0 += 32) {
            int lo, hi;
            range(r0 + lane, lo, hi);
            n += max(0, hi - max(lo, c) + 1);
        }
        return __reduce_add_sync(0xffffffffu, n);
    };
    int c_max = hi0;
    for (int r0 = 32; r0 < a.n_seg; r0 += 32) {
        int lo, hi;
        range(r0 + lane, lo, hi);
        c_max = max(c_max, hi);
    }
    c_max = __reduce_max_sync(0xffffffffu, c_max);
    if (c_max < 1 || jj >= count(1)) return -1;
    int c_lo = 1, c_hi = c_max;  // largest c with count(c) > jj
    while (c_lo < c_hi) {
        const int mid = (c_lo + c_hi + 1) >> 1;
        if (count(mid) > jj) c_lo = mid;
        else c_hi = mid - 1;
    }
    const int c = c_lo;
    int k = jj - (c < c_max ? count(c + 1) : 0);  // rank inside level c
    for (int r0 = 0; r0 < a.n_seg; r0 += 32) {
        int lo = lo0, hi = hi0;
        if (r0 > 0) range(r0 + lane, lo, hi);
        const unsigned has = __ballot_sync(0xffffffffu, lo <= c && c <= hi);
        const int n = __popc(has);
        if (k < n) {
            const int bit = __fns(has, 0, k + 1);
            const int r = r0 + bit;
            const int lo_r = __shfl_sync(0xffffffffu, lo, bit);
            *t = c - lo_r;
            return r;
        }
        k -= n;
    }
    return -1;
}

// Causal prefill, head_dim 128: one CTA per job (query tile t, request b,
// query head h) on the grid (hq, batch, qtiles), blockIdx.x the head.  The
// longest jobs launch first: for the plain prefill the query tile is the
// reversed z index (a job's key tiles grow with it); for the chunked form,
// whose jobs differ by their cached tiles too, the rest of the block index is
// the job in prefill_job's order (most key tiles first, empty slots of the
// grid last).  The query heads of a KV head are adjacent (their K/V tiles
// come from L2 the second time); the hardware scheduler balances the uneven
// jobs, two CTAs per SM.
// The first tiles are requested right after the barriers are set up, before
// the TMEM allocation.
//
// PAST (chunked prefill): request b already holds n_past[b] positions in its
// pages; the job first walks the cached key tiles (positions [128u, 128u +
// 128) < n_past, gathered page by page through the page table with 16-row
// TMA boxes over the pool; every new row sees every cached position), then
// the new key tiles 0..t as below.  Rows of a cached tile past n_past (slots
// of the boundary page that this very launch is writing, or pages not
// loaded) are masked, and their V rows are zeroed in shared memory before
// P V, so stale bits (NaN sentinels included) never meet a zero probability.
//
// Per key tile:
//   - S = Q K^T (Q loaded with the first key tile and kept);
//   - as soon as S has read K, the next key tile's K is requested;
//   - softmax with P_hi and P_lo both in TMEM over the scores
//     (softmax_tile_regs), so no shared memory is written and K stays free
//     for its prefetch;
//   - O += P V with both P terms read from TMEM (issue_pv_tp); when it is
//     done the next key tile's V is requested.
// While the last P V runs, the diagonal tile's (new tile t's) K and V rows go
// to their KV-cache pages at positions n_past + row: the even query head's
// job writes the K rows, the odd one's the V rows (one query head per KV
// head: both), whole pages by TMA stores, the rest by write_kv_pages.  The
// epilogue stages O in the dead Q buffer (store_rows_staged).  TMEM: S/P in
// columns [0, 128), O in [128, 256).
// Cached key tile u of a chunked request (positions [128u, 128u + 128)):
// the K or V rows of pages 8u .. 8u + 7 that hold positions < past, one
// 16-row TMA box per page per 64-dim sub-tile, into the buffer at dst, plus
// the Q tile when with_q; one arrival with the total byte count on bar.  A
// page id outside [0, num_pages) sets QA_DEVICE_BAD_PAGE and is not loaded.
// Page ids [0, n_pre) come from pid_s (shared memory, read once at the start
// of the job), the rest from the page table.  Warp-collective: lane
// kSub * p + sd issues page p's sub-tile sd (and lane sd the Q tile's), so
// the sixteen box requests leave in parallel rather than one after another
// from the thread that also runs a softmax row.
template <int D>
__device__ __forceinline__ void cached_tile_loads(uint32_t sb, uint32_t dst, const CUtensorMap *tm_pool,
                                                  const CUtensorMap *tm_q, bool with_q, int h, int q0,
                                                  const int32_t *pt_row, const int *pid_s, int n_pre, int u,
                                                  int past, int g, int num_pages, uint32_t bar, unsigned int *status) {
    using L = AttnTcLayout<D>;
    static_assert(8 * L::kSub <= 32, "one lane per box");
    const int lane = threadIdx.x & 31;
    const int p = lane / L::kSub, sd = lane % L::kSub;
    int id = -1;
    bool live = p < 8 && 128 * u + 16 * p < past;
    if (live) {
        const int j = 8 * u + p;
        id = j < n_pre ? pid_s[j] : pt_row[j];
        if (id < 0 || id >= num_pages) {
            if (sd == 0) atomicOr(status, QA_DEVICE_BAD_PAGE);
            live = false;
        }
    }
    const unsigned boxes = __ballot_sync(0xffffffffu, live);
    if (lane == 0)
        mbar_arrive_expect_tx(bar, (uint32_t)__popc(boxes) * 16u * 128u + (with_q ? L::kSub * tc::kSubTileBytes : 0u));
    __syncwarp();
    if (live) tc::tma_load_3d(dst + sd * tc::kSubTileBytes + p * 16 * 128, tm_pool, sd * 64, g, id * 16, bar);
    if (with_q && lane < L::kSub)
        tc::tma_load_3d(sb + L::kQ + lane * tc::kSubTileBytes, tm_q, lane * 64, h, q0, bar);
}

template <int GROUP, bool PAST>
__global__ void __launch_bounds__(128, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kp,
                      const __grid_constant__ CUtensorMap tm_vp, const AttnTcArgs a, unsigned int *status) {
    constexpr int D = 128;
    using L = AttnTcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    // launched as a programmatic dependent: wait for the kernel before it
    // (and its writes) before reading anything -- or, when the caller vouches
    // that segments, cached lengths and page table are not its output
    // (a.early), only before the first tile loads -- then let the next kernel
    // be scheduled once every CTA of this grid has started
    if (!a.early) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }

    const int h = blockIdx.x, g = h / GROUP;
    const int max_len = a.max_pages * a.page_size;
    int b, qt;
    if (PAST) {
        // chunked form: jobs differ by their cached tiles too, so the rest
        // of the block index is the job in prefill_job's order
        const int jj = (int)(blockIdx.y + gridDim.y * blockIdx.z);
        volatile int *job = reinterpret_cast<volatile int *>(smem + L::kNext);
        if (warp == 0) {
            const int lane = tid & 31;
            if (jj == 0 && h == 0) {
                // the first CTA checks every request once: segments, cached
                // lengths, and requests longer than their page-table row
                // (clipped: rows past the row's capacity are neither written
                // nor, beyond the grid, attended)
                bool bad_seg = a.cu[a.n_seg] != a.total, bad_len = false;
                for (int r = lane; r < a.n_seg; r += 32) {
                    const int r0 = a.cu[r], r1 = a.cu[r + 1], pst = a.n_past[r];
                    bad_seg |= !(0 <= r0 && r0 <= r1 && r1 <= a.total);
                    bad_len |= pst < 0 || pst > max_len || (a.k_pages && r1 - r0 > max_len - pst);
                }
                const bool any_seg = __any_sync(0xffffffffu, bad_seg), any_len = __any_sync(0xffffffffu, bad_len);
                if (lane == 0 && any_seg) atomicOr(status, QA_DEVICE_BAD_SEGMENTS);
                if (lane == 0 && any_len) atomicOr(status, QA_DEVICE_BAD_LENGTH);
            }
            int t = 0;
            const int bb = prefill_job(a, true, jj, (int)gridDim.z, max_len, &t);  // gridDim.z: tiles of a row
            if (lane == 0) {
                job[0] = bb;
                job[1] = t;
            }
        }
        __syncthreads();
        b = job[0];
        qt = job[1];
        if (b < 0 || a.cu[a.n_seg] != a.total) return;
    } else {
        // the query tile reversed: the last query tiles (the most key tiles)
        // launch first
        b = blockIdx.y;
        qt = (int)(gridDim.z - 1 - blockIdx.z);
    }
    const int s0 = a.cu[b], s1 = a.cu[b + 1];
    if (!(0 <= s0 && s0 <= s1 && s1 <= a.total) || a.cu[a.n_seg] != a.total) {
        if (!PAST && tid == 0) atomicOr(status, QA_DEVICE_BAD_SEGMENTS);
        return;
    }
    const int past = PAST ? a.n_past[b] : 0;
    if (PAST && (past < 0 || past > max_len)) return;
    // a request longer than its page-table row: flagged once; its rows past
    // the row's capacity are neither written nor (beyond the grid) attended
    if (!PAST && a.k_pages && qt == 0 && h == 0 && tid == 0 && s1 - s0 > max_len)
        atomicOr(status, QA_DEVICE_BAD_LENGTH);
    if (qt * 128 >= s1 - s0) return;
    const int q0 = s0 + qt * 128;
    const int n_ct = PAST ? (past + 127) / 128 : 0;  // cached key tiles
    const int n_tiles = n_ct + qt + 1;
    const int32_t *pt_row = a.page_table + (size_t)b * a.max_pages;

    const uint32_t bar_k = sb + L::kBar, bar_s = bar_k + 8, bar_o = bar_k + 16, bar_v = bar_k + 24;
    // chunked form: the page ids of the cached positions (up to kPre of
    // them), read by warp 0 once so that the cached tiles' loads do not wait
    // on the page table each time
    constexpr int kPre = 256;
    int *pid_s = reinterpret_cast<int *>(smem + L::kBytes);
    const int n_pre = PAST ? min(kPre, (past + 15) / 16) : 0;
    if (PAST && warp == 0) {
        for (int j = tid; j < n_pre; j += 32) pid_s[j] = pt_row[j];
        __syncwarp();
    }
    // warp 0: requests the K (with Q for the first tile) or V tile of key
    // tile u (a cached tile's boxes leave from its lanes, a new tile's from
    // lane 0)
    auto load_k = [&](int u, bool with_q) {
        if (PAST && u < n_ct)
            cached_tile_loads<D>(sb, sb + L::kK, &tm_kp, &tm_q, with_q, h, q0, pt_row, pid_s, n_pre, u, past, g,
                                 a.num_pages, bar_k, status);
        else if (tid == 0)
            issue_qk_loads<D>(sb, &tm_q, &tm_k, h, g, q0, s0 + (u - n_ct) * 128, with_q, bar_k);
    };
    auto load_v = [&](int u) {
        if (PAST && u < n_ct)
            cached_tile_loads<D>(sb, sb + L::kV, &tm_vp, &tm_q, false, h, q0, pt_row, pid_s, n_pre, u, past, g,
                                 a.num_pages, bar_v, status);
        else if (tid == 0)
            issue_v_loads<D>(sb, &tm_v, g, s0 + (u - n_ct) * 128, bar_v);
    };
    if (tid == 0) {
        mbar_init(bar_k, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
    }
    if (warp == 0 && !a.early) {
        __syncwarp();  // the barriers are set up
        load_k(0, true);
        load_v(0);
    }
    if (warp == 0) tc::tmem_alloc(sb + L::kTmemSlot, 256);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (a.early) {  // the job is set up; q, k, v, the pools and out only now
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (warp == 0) {
            load_k(0, true);
            load_v(0);
        }
    }
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t col_o = 128;
    uint32_t ph = 0;  // every barrier completes once per key tile
    const int li = qt * 128 + tid;  // local index of this thread's new row
    float m = -INFINITY, l = 0.f;
    // page write of the diagonal tile (the last one): with two query heads
    // per KV head, the even head's CTA writes the K rows and the odd one the
    // V rows (both hold the same tiles); the page ids are read now, long
    // before they are needed
    const bool write_k = a.k_pages && h % GROUP == 0;
    const bool write_v = a.k_pages && (GROUP == 1 || h % GROUP == 1);
    const int my_page = (write_k || write_v) ? kv_tile_page_id(a, b, qt * 128, s1 - s0, past, tid) : -1;

    for (int u = 0; u < n_tiles; ++u, ph ^= 1) {
        const bool cached = PAST && u < n_ct;
        const int kt = u - n_ct;  // new key tile (when not cached)
        if (tid == 0) {
            mbar_wait(bar_k, ph, status);
            tc::fence_after();
            issue_s<D>(tmem, sb + L::kQ, sb + L::kK);
            tc::mma_commit(bar_s);
        }
        mbar_wait(bar_s, ph, status);
        tc::fence_after();
        // S has read K: the next key tile's K
        if (warp == 0 && u + 1 < n_tiles) load_k(u + 1, false);
        int n_ok;
        if (cached) {
            // every cached position before `past` is visible to every new row
            n_ok = min(128, past - 128 * u);
            if (n_ok < 128) {
                // rows past n_ok: stale or in-flight bits; zero their V rows
                mbar_wait(bar_v, ph, status);
                if (tid >= n_ok) {
#pragma unroll
                    for (int sd = 0; sd < L::kSub; ++sd)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            tc::st_shared_v4(sb + L::kV + sd * tc::kSubTileBytes + tid * 128 + c * 16, 0u, 0u, 0u, 0u);
                }
                tc::fence_proxy_async_smem();
            }
        } else {
            n_ok = min(128, (s1 - s0) - 128 * kt);
            n_ok = min(n_ok, li - 128 * kt + 1);
            n_ok = max(n_ok, 0);
        }
        // P V in two halves of 64 keys: the first starts as soon as every
        // row has written P for keys [0, 64), the second after the softmax
        softmax_tile_regs<D>(t_row, n_ok, a.scale_log2, t_row + col_o, u > 0, m, l, [&] {
            tc::tmem_wait_st();
            tc::fence_before();
            __syncthreads();
            if (tid == 0) {
                mbar_wait(bar_v, ph, status);
                tc::fence_after();
                issue_pv_tp<D>(tmem, tmem + col_o, sb + L::kV, u > 0, 0);
            }
        });
        tc::fence_before();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after();
            issue_pv_tp<D>(tmem, tmem + col_o, sb + L::kV, true, 1);
            tc::mma_commit(bar_o);
        }
        if (u == n_tiles - 1 && (write_k || write_v)) {
            // diagonal tile: its K/V rows are this query tile's own; written
            // while the last P V runs (both only read the tiles).  Whole
            // pages (the tile's rows start a page when past is a multiple of
            // 16) go out as 16-row TMA stores through the pool maps, one per
            // page and 64-dim sub-tile, issued by lane j of warp 0 for the
            // j-th page; the rows of a partial last page, or every row when
            // the tile does not start a page, with plain stores.
            mbar_wait(bar_v, ph, status);
            const int end = min(min(s1 - s0, max_len - past) - qt * 128, 128);
            const int tma_rows = (past % 16 == 0 && end > 0) ? end / 16 * 16 : 0;
            if (warp == 0 && (tid & 31) < tma_rows / 16) {
                if (my_page < 0 || my_page >= a.num_pages) {
                    atomicOr(status, QA_DEVICE_BAD_PAGE);
                } else {
                    const uint32_t row_off = (uint32_t)(tid & 31) * 16u * 128u;
#pragma unroll
                    for (int sd = 0; sd < L::kSub; ++sd) {
                        if (write_k)
                            tc::tma_store_3d(&tm_kp, sb + L::kK + sd * tc::kSubTileBytes + row_off, sd * 64, g,
                                             my_page * 16);
                        if (write_v)
                            tc::tma_store_3d(&tm_vp, sb + L::kV + sd * tc::kSubTileBytes + row_off, sd * 64, g,
                                             my_page * 16);
                    }
                    tc::bulk_commit_group();
                }
            }
            if (tma_rows < end)
                write_kv_pages<D>(write_k ? smem + L::kK : nullptr, write_v ? smem + L::kV : nullptr, a, qt * 128,
                                  s1 - s0, past, g, status, tid, my_page, tma_rows);
        }
        mbar_wait(bar_o, ph, status);
        tc::fence_after();
        if (warp == 0 && u + 1 < n_tiles) load_v(u + 1);
    }
    // staged in the dead Q buffer (the page write may still read K and V)
    store_rows_staged<D>(t_row + col_o, l, sb + L::kQ, a.out, a.hq, h, q0, min(128, s1 - q0), tid);
    if (warp == 0) tc::bulk_wait_group_read_all();  // the TMA page stores have read K and V
    tc::fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 256);
    }
}

}  // namespace qa
