// Dense projections of the AuT encoder layer on the tensor cores:
//
//   out[m][n] = act(sum_k A[m][k] W[n][k] + bias[n]) + res[m][n]
//
// A [M][K] bf16 row-major (activations), W [N][K] bf16 (a PyTorch Linear
// weight, qwenasr.cpp ARCHITECTURE.md "Tensor shape and layout": (out, in),
// y = x W^T), bias [N] bf16 or none, act none or the exact gelu
// u / 2 (1 + erf(u / sqrt 2)) ("Windowed audio tower": gelu MLP; "GGML
// conventions": ggml_gelu_erf), res [M][N] bf16 (the residual stream) or
// none.  fp32 accumulation, bf16 result (round to nearest even) with any row
// stride, so the fused q|k|v projection writes one [M][3 d] buffer.
//
// Persistent, warp-specialised, one CTA per SM, the CTAs in pairs (clusters
// of two on two SMs) that share one 256 x BN output tile: rank r of the pair
// holds rows [128 r, 128 r + 128) of the tile's A block and W rows
// [BN / 2 r, BN / 2 (r + 1)) of its W block, and one tcgen05.mma.cta_group::2
// (M = 256) reads both CTAs' halves and writes each CTA's 128 rows of the
// accumulator into that CTA's TMEM -- so an SM takes in 16 KiB of A and
// BN / 2 x 128 bytes of W per 64-wide K step instead of the whole W tile:
//   warp 0     producer (both CTAs): TMA loads of its 128 x 64 A tile and its
//              BN / 2 x 64 W half (128-byte swizzled, K-major) into a ring of
//              shared-memory stages; both CTAs' loads of a stage complete on
//              rank 0's "full" mbarrier, whose producer expects the bytes of
//              both;
//   warp 1     allocates the pair's TMEM; on rank 0 one lane issues the MMAs
//              (K = 16 per instruction, four per 64-wide stage) into one of two
//              fp32 accumulators; a stage is released ("empty") in both CTAs
//              by a multicast tcgen05.commit when its MMAs are done, and an
//              accumulator is handed to both epilogues ("acc_full") the same
//              way;
//   warps 2-9  epilogue (both CTAs), two warpgroups splitting the tile's
//              columns: each thread owns one row of its CTA's 128 rows (the
//              TMEM lane quadrant of its warp), reads the accumulator 32
//              columns at a time, adds bias, applies gelu, adds the residual
//              (its 32 x 32 block brought in by TMA one chunk ahead), rounds
//              to bf16 into a staging block that one lane writes out with a
//              TMA store; then releases the accumulator on rank 0's
//              "acc_empty" barrier so the next-but-one tile can use it.
// With two accumulators the epilogue of tile i overlaps the MMAs of tile
// i + 1.  Tiles are walked m-block-major (tile = m_blk * tiles_n + n_blk), so
// the pairs running at any moment share a few m-blocks of A and every W tile:
// A is fetched from HBM about once, W stays in L2.
//
// Rows past M and columns past N (ragged last tiles) are zero-filled by the
// TMA loads and clipped by the TMA stores; K need not be a multiple of 64 (the zero fill makes the
// tail products 0).  Every wait is bounded (common.cuh): one that expires
// sets QA_DEVICE_TIMEOUT and the kernel runs to its end.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "qa_internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace qa {
namespace {

__device__ unsigned int g_status;

constexpr int kBM = 128, kBK = 64;  // rows of A per CTA (256 per pair), K step
constexpr int kEpiWarps = 8;  // two epilogue warpgroups, each covering all 128 TMEM lanes
constexpr int kThreads = 32 * (2 + kEpiWarps);  // producer, MMA, epilogue

struct GemmArgs {
    int M, N, K;
    const uint16_t *bias;  // [N] or null
    const uint16_t *res;   // [M][ldr] or null
    uint16_t *out;         // [M][ldc]
    long long ldr, ldc;
    int act;  // 0 none, 1 gelu (erf)
    int tiles_m, tiles_n;
};

template <int BN, bool RES>
struct GemmLayout {
    static constexpr uint32_t kA = kBM * kBK * 2;        // 16 KiB
    static constexpr uint32_t kB = (BN / 2) * kBK * 2;   // this CTA's half of the W tile
    static constexpr uint32_t kStage = kA + kB;
    // epilogue staging, per epilogue warp: two 32 x 32 output blocks and, with
    // a residual, two 32 x 32 residual blocks of bf16 (2 KiB each, 64-byte
    // swizzled)
    static constexpr uint32_t kEpiWarpBytes = (RES ? 4 : 2) * 2048;
    static constexpr uint32_t kEpiBytes = kEpiWarps * kEpiWarpBytes;
    static constexpr int kStages = (220 * 1024 - kEpiBytes) / kStage < 8 ? (220 * 1024 - kEpiBytes) / kStage : 8;
    static constexpr uint32_t kEpi = kStages * kStage;
    // full[S], empty[S], acc_full[2], acc_empty[2], then two residual
    // barriers per epilogue warp
    static constexpr uint32_t kBar = kEpi + kEpiBytes;
    static constexpr uint32_t kResBar = kBar + (2 * kStages + 4) * 8;
    static constexpr uint32_t kTmemSlot = kResBar + kEpiWarps * 2 * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 8;  // set when a wait expired: every role stops
    static constexpr uint32_t kBytes = kTmemSlot + 16;
    static constexpr uint32_t kSmem = kBytes + 1024;  // slack for 1024-byte alignment
    static constexpr uint32_t kAccCols = 256;         // column stride of the two accumulators
    static_assert(kA % 1024 == 0 && kB % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "N tile: a multiple of 32, at most 256");
    static_assert(kStages >= 2, "at least two stages");
    static_assert(kSmem <= 227 * 1024, "shared memory");
};

// gelu(u) = u / 2 (1 + erf(u / sqrt 2)), with erf from Abramowitz and Stegun,
// Handbook of Mathematical Functions, formula 7.1.26: for z >= 0,
// erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2) with
// t = 1 / (1 + p z), absolute error at most 1.5e-7 (odd in z) -- far below
// the bf16 rounding of the result (the approximate reciprocal and exp2 add a
// few ulps of fp32).  Two MUFU operations and a handful of FMAs per element.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Two elements at once on packed fp32 pairs, written as
// gelu(u) = max(u, 0) - |u| / 2 * Q(|u| / sqrt 2), Q(z) = 1 - erf(z) =
// (a1 t + ... + a5 t^5) exp(-z^2) from the same formula (no cancellation in
// 1 - Q for negative u).
__device__ __forceinline__ float2 gelu_erf2(float2 u) {
    const float2 a = make_float2(fabsf(u.x), fabsf(u.y));
    const float2 z = fmul2(a, make_float2(0.70710678118654752f, 0.70710678118654752f));
    const float2 d = ffma2(z, make_float2(0.3275911f, 0.3275911f), make_float2(1.0f, 1.0f));  // 1 + p z >= 1
    const float2 t = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    float2 poly = ffma2(make_float2(1.061405429f, 1.061405429f), t, make_float2(-1.453152027f, -1.453152027f));
    poly = ffma2(poly, t, make_float2(1.421413741f, 1.421413741f));
    poly = ffma2(poly, t, make_float2(-0.284496736f, -0.284496736f));
    poly = ffma2(poly, t, make_float2(0.254829592f, 0.254829592f));
    poly = fmul2(poly, t);
    const float2 x = fmul2(z, fmul2(z, make_float2(-kLog2e, -kLog2e)));  // -z^2 log2(e)
    const float2 q = fmul2(poly, make_float2(exp2_approx(x.x), exp2_approx(x.y)));
    return ffma2(fmul2(a, make_float2(-0.5f, -0.5f)), q, make_float2(fmaxf(u.x, 0.f), fmaxf(u.y, 0.f)));
}

// bf16x8 (one 16-byte word) -> 8 floats
__device__ __forceinline__ void unpack8(uint4 w, float *f) {
    f[0] = bf16lo(w.x), f[1] = bf16hi(w.x), f[2] = bf16lo(w.y), f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z), f[5] = bf16hi(w.z), f[6] = bf16lo(w.w), f[7] = bf16hi(w.w);
}

template <int BN, bool RES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_res,
                     const GemmArgs a) {
    using L = GemmLayout<BN, RES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank();  // 0: issues the pair's MMAs
    const uint32_t bar_full = sb + L::kBar, bar_empty = bar_full + L::kStages * 8;
    const uint32_t bar_acc_full = bar_empty + L::kStages * 8, bar_acc_empty = bar_acc_full + 16;
    const int n_tiles = a.tiles_m * a.tiles_n;  // 256-row tiles
    const int n_kb = (a.K + kBK - 1) / kBK;
    const int pair = (int)blockIdx.x >> 1, n_pairs = (int)gridDim.x >> 1;

    // a programmatic dependent of the kernel before it: wait for its writes
    // before reading anything, then let the next kernel be scheduled
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        *reinterpret_cast<volatile int *>(smem + L::kAbort) = 0;
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);   // rank 0's: its producer's arrival (both CTAs' bytes)
            mbar_init(bar_empty + 8 * s, 1);  // the MMA thread's multicast commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_acc_full + 8 * i, 1);
            mbar_init(bar_acc_empty + 8 * i, 2 * kEpiWarps);  // rank 0's: every epilogue warp of the pair
        }
        for (int i = 0; i < 2 * kEpiWarps; ++i) mbar_init(sb + L::kResBar + 8 * i, 1);
        fence_mbar_init();
        tc::prefetch_tmap(&tm_a);
        tc::prefetch_tmap(&tm_w);
        tc::prefetch_tmap(&tm_out);
        if (RES) tc::prefetch_tmap(&tm_res);
    }
    if (warp == 1) tc::tmem_alloc_pair(sb + L::kTmemSlot, 512);
    tc::fence_before();
    tc::cluster_sync();  // both CTAs' barriers are set up before either signals the other's
    tc::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    // A wait that expires (a fault elsewhere) stops every role of this CTA
    // at its next wait instead of letting each later wait expire in turn.
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbort);
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity, &g_status)) return true;
        *abort_flag = 1;
        return false;
    };
    const uint32_t full0 = tc::map_to_rank(bar_full, 0);            // rank 0's full barriers
    const uint32_t acc_empty0 = tc::map_to_rank(bar_acc_empty, 0);  // rank 0's acc_empty barriers

    if (warp == 0) {
        // ---------------- producer (both CTAs): this CTA's A rows and W half
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = pair; tile < n_tiles && ok; tile += n_pairs) {
                const int m0 = (tile / a.tiles_n) * (2 * kBM) + (int)rank * kBM;
                const int n0 = (tile % a.tiles_n) * BN + (int)rank * (BN / 2);
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % L::kStages;
                    if (it >= L::kStages && !(ok = wait(bar_empty + 8 * s, ((it / L::kStages) & 1) ^ 1))) break;
                    const uint32_t st = sb + s * L::kStage;
                    // rank 0 expects the bytes of both CTAs' loads; rank 1's
                    // loads only count theirs on rank 0's barrier (a stage is
                    // refilled only after the MMAs that read it, so no count
                    // from the next round can meet the current one)
                    if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * L::kStage);
                    tc::tma_load_2d_pair(st, &tm_a, kb * kBK, m0, full0 + 8 * s);
                    tc::tma_load_2d_pair(st + L::kA, &tm_w, kb * kBK, n0, full0 + 8 * s);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issue (rank 0 only)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16(2 * kBM, BN, false);
            int it = 0, tcount = 0;
            bool ok = true;
            for (int tile = pair; tile < n_tiles && ok; tile += n_pairs, ++tcount) {
                const int acc = tcount & 1;
                if (tcount >= 2 && !(ok = wait(bar_acc_empty + 8 * acc, ((tcount >> 1) & 1) ^ 1))) break;
                tc::fence_after();
                const uint32_t d_tmem = tmem + acc * L::kAccCols;
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % L::kStages;
                    if (!(ok = wait(bar_full + 8 * s, (it / L::kStages) & 1))) break;
                    tc::fence_after();
                    const uint32_t st = sb + s * L::kStage;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_bf16_pair(d_tmem, tc::sw128_desc(st + kk * 32), tc::sw128_desc(st + L::kA + kk * 32),
                                          idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    tc::mma_commit_pair(bar_empty + 8 * s);  // the stage is free (both CTAs) once these are done
                }
                if (ok) tc::mma_commit_pair(bar_acc_full + 8 * acc);
            }
        }
    } else {
        // ---------------- epilogue (both CTAs): warps 2..9, TMEM lane
        // quadrant warp % 4; warpgroup eg = 0 takes the first half of the
        // tile's 32-column chunks, eg = 1 the rest.  A warp's 32 rows of a
        // chunk form one 32 x 32 block: the residual block comes in by TMA
        // (one chunk ahead, the first before the wait for the accumulator)
        // and the output block leaves by a TMA store from a staging block,
        // so no thread waits on a global load or issues a scattered store.
        // The blocks are 64-byte swizzled: 16-byte chunk k of row r sits at
        // chunk position k ^ ((r / 2) % 4), which spreads a warp's row
        // accesses over every bank.
        const int quad = warp & 3;
        const int ew = warp - 2;
        const int eg = ew >> 2;
        constexpr int kChunks = BN / 32;
        const int c_begin = eg == 0 ? 0 : (kChunks + 1) / 2, c_end = eg == 0 ? (kChunks + 1) / 2 : kChunks;
        const uint32_t ostage = sb + L::kEpi + (uint32_t)ew * L::kEpiWarpBytes;  // two output blocks
        const uint32_t rstage = ostage + 2 * 2048;                               // two residual blocks
        const uint32_t bar_res = sb + L::kResBar + (uint32_t)ew * 16;
        const uint32_t sw = (uint32_t)((lane >> 1) & 3);
        const uint32_t orow = (uint32_t)lane * 64u;
        uint32_t res_phase = 0;  // bit b: parity of residual block b's next completion
        int kc = 0;              // chunks this warp has handled (block index kc & 1)
        // bias words of chunk c (8 bf16 per word), loaded one chunk ahead
        auto bias_loads = [&](int n0, int c, uint4 (&bw)[4]) {
            const int col0 = n0 + c * 32;
            const int n_groups = max(0, min(4, (a.N - col0) / 8));  // 8-column groups inside N
#pragma unroll
            for (int g = 0; g < 4; ++g)
                bw[g] = (a.bias && g < n_groups) ? *reinterpret_cast<const uint4 *>(a.bias + col0 + 8 * g)
                                                 : make_uint4(0u, 0u, 0u, 0u);
        };
        auto res_load = [&](int n0, int row0, int c, int blk) {
            if (RES && lane == 0) {
                mbar_arrive_expect_tx(bar_res + 8 * blk, 2048);
                tc::tma_load_2d(rstage + (uint32_t)blk * 2048, &tm_res, n0 + 32 * c, row0, bar_res + 8 * blk);
            }
        };
        int tcount = 0;
        for (int tile = pair; tile < n_tiles; tile += n_pairs, ++tcount) {
            const int acc = tcount & 1;
            const int m0 = (tile / a.tiles_n) * (2 * kBM), n0 = (tile % a.tiles_n) * BN;
            const int row0 = m0 + (int)rank * kBM + quad * 32;  // the warp's first row
            uint4 bw[4];
            bias_loads(n0, c_begin, bw);
            res_load(n0, row0, c_begin, kc & 1);
            // warp-uniform: every lane waits on the same phase
            const bool ok = wait(bar_acc_full + 8 * acc, (tcount >> 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after();
            const uint32_t t_base = tmem + acc * L::kAccCols + ((uint32_t)(quad * 32) << 16);
#pragma unroll 1
            for (int c = c_begin; c < c_end; ++c, ++kc) {
                const int blk = kc & 1;
                uint4 nbw[4] = {};
                if (c + 1 < c_end) {
                    bias_loads(n0, c + 1, nbw);
                    res_load(n0, row0, c + 1, blk ^ 1);  // that block was read in the previous chunk
                }
                float v[32];
                tc::tmem_ld32(t_base + c * 32, v);  // warp-collective: every lane, every chunk
                float rf[32] = {};
                if (RES) {
                    wait(bar_res + 8 * blk, (res_phase >> blk) & 1);
                    res_phase ^= 1u << blk;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t x0, x1, x2, x3;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                                     : "r"(rstage + (uint32_t)blk * 2048 + orow + (((uint32_t)k ^ sw) << 4)));
                        unpack8(make_uint4(x0, x1, x2, x3), rf + 8 * k);
                    }
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float bf[8];
                    unpack8(bw[g], bf);
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        float2 u = fadd2(make_float2(v[8 * g + j], v[8 * g + j + 1]), make_float2(bf[j], bf[j + 1]));
                        if (a.act == 1) u = gelu_erf2(u);
                        if (RES) u = fadd2(u, make_float2(rf[8 * g + j], rf[8 * g + j + 1]));
                        v[8 * g + j] = u.x;
                        v[8 * g + j + 1] = u.y;
                    }
                }
                // the output block written two chunks ago has been read by
                // its TMA store before this one overwrites it
                if (lane == 0) tc::bulk_wait_group_read_1();
                __syncwarp();
                const uint32_t ob = ostage + (uint32_t)blk * 2048 + orow;
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    tc::st_shared_v4(ob + (((uint32_t)g ^ sw) << 4), pack_bf16x2(v[8 * g + 0], v[8 * g + 1]),
                                     pack_bf16x2(v[8 * g + 2], v[8 * g + 3]), pack_bf16x2(v[8 * g + 4], v[8 * g + 5]),
                                     pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
                tc::fence_proxy_async_smem();  // the block is read by the TMA unit
                __syncwarp();
                // rows past M and columns past N are clipped by the store
                if (lane == 0) {
                    tc::tma_store_2d(&tm_out, ostage + (uint32_t)blk * 2048, n0 + 32 * c, row0);
                    tc::bulk_commit_group();
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) bw[g] = nbw[g];
            }
            // every TMEM read of this accumulator is done: hand it back to
            // the MMA thread (on rank 0)
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(acc_empty0 + 8 * acc);
        }
        if (lane == 0) tc::bulk_wait_group_read_all();  // the stores have read their blocks
    }

    __syncwarp();  // lanes 1..31 of the producer and MMA warps wait for their lane 0
    if (*abort_flag && warp == 0 && lane == 0) {
        // a wait expired: give the loads this CTA issued (whose completion is
        // counted on rank 0's barriers) 100 us to land before its shared
        // memory is given up
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 100000ull) {
        }
    }
    tc::fence_before();
    // both CTAs are done: rank 0's MMAs no longer read rank 1's shared memory,
    // and no arrival on rank 0's barriers is still on its way
    tc::cluster_sync();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc_pair(tmem, 512);
    }
}

// 2-D tensor map of a row-major bf16 matrix [rows][cols] with row stride ld
// (elements): box {64 cols, box_rows rows}, 128-byte swizzle.
bool make_matrix_tmap(CUtensorMap *map, const void *base, long long rows, long long cols, long long ld,
                      int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || rows < 1 || cols < 1 || rows > 0x7fffffffLL || cols > 0x7fffffffLL) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D tensor map of a row-major bf16 matrix [rows][cols] with row stride ld
// (elements, a multiple of 8): box {32 cols, 32 rows}, 64-byte swizzle (the
// epilogue's blocks).
bool make_block_tmap(CUtensorMap *map, const void *base, long long rows, long long cols, long long ld) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || rows < 1 || cols < 1 || rows > 0x7fffffffLL || cols > 0x7fffffffLL) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, bool RES>
cudaError_t launch_gemm_bn(const void *x, long long ldx, int M, int K, const void *w, int N, const void *bias,
                           int act, const void *res, long long ldr, void *out, long long ldc, cudaStream_t stream) {
    using L = GemmLayout<BN, RES>;
    CUtensorMap ta, tw, tout, tres;
    // each CTA of a pair loads 128 rows of A and BN / 2 rows of W; the
    // epilogue moves 32 x 32 blocks of the output and the residual
    if (!make_matrix_tmap(&ta, x, M, K, ldx, kBM) || !make_matrix_tmap(&tw, w, N, K, K, BN / 2) ||
        !make_block_tmap(&tout, out, M, N, ldc) || (res && !make_block_tmap(&tres, res, M, N, ldr)))
        return cudaErrorInvalidValue;
    if (!res) tres = tout;  // not read
    GemmArgs a{};
    a.M = M, a.N = N, a.K = K;
    a.bias = static_cast<const uint16_t *>(bias);
    a.res = static_cast<const uint16_t *>(res);
    a.out = static_cast<uint16_t *>(out);
    a.ldr = ldr, a.ldc = ldc, a.act = act;
    a.tiles_m = (M + 2 * kBM - 1) / (2 * kBM);
    a.tiles_n = (N + BN - 1) / BN;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_bf16_kernel<BN, RES>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    const long long tiles = (long long)a.tiles_m * a.tiles_n;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // Persistent: as many pairs as can be resident at once (an SM whose
    // partner SM is disabled hosts no pair, so this is below sms / 2; more
    // pairs than fit would run as a second wave), cached per device.
    static int max_pairs[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (max_pairs[dev] == 0) {
        int n = 0;
        cfg.gridDim = dim3((unsigned)(2 * std::max(1, sms / 2)));
        e = cudaOccupancyMaxActiveClusters(&n, gemm_bf16_kernel<BN, RES>, &cfg);
        if (e != cudaSuccess) return e;
        max_pairs[dev] = std::max(1, n);
    }
    const long long pairs = std::min<long long>(tiles, max_pairs[dev]);
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    e = cudaLaunchKernelEx(&cfg, gemm_bf16_kernel<BN, RES>, ta, tw, tout, tres, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

// N tile: 256 where it divides N (per flop, fewer A bytes through L2 than
// 224, and both epilogue warpgroups take four 32-column chunks of a tile;
// fc1's 3584: 305 us instead of 324); else 224 where that divides N exactly
// (the encoder's 896 and 3 x 896); else 256 with a ragged last tile.
cudaError_t launch_gemm(const void *x, long long ldx, int M, int K, const void *w, int N, const void *bias, int act,
                        const void *res, long long ldr, void *out, long long ldc, cudaStream_t stream) {
    if (M == 0) return cudaSuccess;
    if (N % 256 != 0 && N % 224 == 0)
        return res ? launch_gemm_bn<224, true>(x, ldx, M, K, w, N, bias, act, res, ldr, out, ldc, stream)
                   : launch_gemm_bn<224, false>(x, ldx, M, K, w, N, bias, act, res, ldr, out, ldc, stream);
    return res ? launch_gemm_bn<256, true>(x, ldx, M, K, w, N, bias, act, res, ldr, out, ldc, stream)
               : launch_gemm_bn<256, false>(x, ldx, M, K, w, N, bias, act, res, ldr, out, ldc, stream);
}

unsigned int status_read_clear_gemm(cudaStream_t stream, cudaError_t *err) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && v)
        e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (err) *err = e;
    return v;
}

}  // namespace qa
