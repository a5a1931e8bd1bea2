// gemm.cu -- grouped expert matmuls on the 5th-generation tensor cores.
//
// "NPU HunyuanImage-3.0模型推理优化实践": "GMM使能&&Routing优化" (one grouped
// matmul computes all experts instead of a per-expert loop) and
// "MoE TP优化 / 计算分解" (gate and up merged into w13; SwiGLU returns
// SiLU(first half) * second half).
//
// One persistent kernel serves both matmuls of the expert FFN:
//   SWIGLU: act[r, n] = bf16(SiLU(g) * u), g = A[r] . W[grp, n], u = A[r] . W[grp, half + n]
//   STORE:  out[r, n] = A[r] . W[grp, n]          (bf16, or fp32 per segment)
// over ragged groups: group g owns rows [offsets[g], offsets[g+1]) of A and
// weight slice W[g].  An optional dense "segment 1" (the shared expert, its
// own A, W and output) is appended to the same tile list.
//
// Tiles are 128 rows x BN columns (SWIGLU: 128 gate + 128 up columns giving
// 128 act columns).  The tile list is built on the device from `offsets`
// (no host sync): per group ceil(rows/128) m-blocks x n-blocks, ordered so
// that CTAs running at the same time share the larger operand through L2
// (m fastest when the group has fewer rows than its weight slice, n fastest
// otherwise, e.g. the shared expert or a very busy expert).  A tile may
// read rows of the next group; the epilogue stores only the group's rows.
//
// CTA roles (192 threads, one CTA per SM):
//   warp 0     TMA producer: A and B k-slices (64 wide, 128-byte swizzle)
//              into a 4-stage shared-memory ring;
//   warp 1     allocates 2*BN TMEM columns; one thread issues
//              tcgen05.mma (M=128, N=BN, K=16) into one of two TMEM
//              accumulators and commits stage releases / tile completion;
//   warps 2-5  epilogue: tcgen05.ld of the finished accumulator (each warp
//              its 32-lane quarter), SwiGLU or conversion, 16-byte stores.
// The two accumulators let the epilogue of tile i overlap the MMAs of i+1.
// Every wait is bounded (MOE_DEV_TIMEOUT) and on abort each role lets its
// in-flight copies / MMAs finish before the TMEM is freed.
//
// Two CTA-pair kernels (tcgen05 cta_group::2, clusters of two SMs, tiles
// handed out in order through a per-launch counter) take the launches with
// many rows per group: 256 x 256 tiles with a double-buffered accumulator,
// and (the default there) 256 x 512 tiles whose accumulator fills TMEM,
// with a quarter fewer operand bytes per flop.  The latter can also copy its
// A rows itself by source token instead of reading permuted rows.  Each is
// described above its code; the host picks per launch (MOE_GEMM_KERNEL=
// single|pair|wide forces one).
#include <cuda.h>

#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;
constexpr int MAX_GROUPS = 1024;

enum { MODE_SWIGLU = 0, MODE_STORE = 1 };

struct Params {
    CUtensorMap tmA0;   // routed A [rows0, K0]
    CUtensorMap tmB0;   // routed W [G, NW0, K0]
    CUtensorMap tmA1;   // segment-1 A [rows1, K1]
    CUtensorMap tmB1;   // segment-1 W [NW1, K1]
    const int32_t *offsets;
    int32_t G;
    int32_t rows0;      // rows of A0 / out0 (bounds the offsets)
    int32_t K0, K1;
    int32_t nt0, nt1;   // n-blocks per m-block
    int32_t half0, half1;
    int32_t brows0, brows1;  // rows of one group's weight slice (2N for SwiGLU, N for store)
    int32_t rows1;      // 0 = no segment 1
    void *out0;
    int64_t ldo0;
    void *out1;
    int64_t ldo1;
    int32_t out0_f32;   // store mode: routed output in fp32 (else bf16)
    int32_t out1_f32;
    int32_t *dev_status;
    unsigned int *tile_counter;   // pair kernel: next tile to hand out (zeroed per launch)
    CUtensorMap tmO0;   // pair kernel: segment-0 output, 32-row x 64-byte boxes, 64-byte swizzle
    CUtensorMap tmO1;   // pair kernel: segment-1 output (bf16 or fp32)
    // pair kernel, half tiles: the same tensors as 64-row boxes (A of both
    // segments; B of the SwiGLU mode, whose half tiles take 64 gate + 64 up rows)
    CUtensorMap tmA0h, tmA1h, tmB0h, tmB1h;
    // wide pair kernel: B of both segments as 256-row boxes
    CUtensorMap tmB0w, tmB1w;
    // wide pair kernel with gathered A (SwiGLU): routed row r is row
    // ga_rows0[r] of gA0 (clamped into its ga_n0 rows), segment-1 row r is
    // row r of gA1; both row-major with K0 / K1 columns
    const uint16_t *gA0;
    const int32_t *ga_rows0;
    int32_t ga_n0;
    const uint16_t *gA1;
};

struct Tile {
    int seg, g, row0, row_end, n_blk, kblocks;
    bool half;   // pair kernel: at most 128 rows left -> an M=128 pair MMA
};

template <int BN>
struct Cfg {
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    // barriers: full[S], empty[S], tfull[2], tempty[2], drain
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int OFFS_OFF = MISC_OFF + 16;
    static constexpr int PREFIX_OFF = OFFS_OFF + (MAX_GROUPS + 1) * 4;
    static constexpr int SMEM = 1024 + PREFIX_OFF + (MAX_GROUPS + 2) * 4;
};

__device__ __forceinline__ Tile decode_tile(const Params &p, int tile, const int *s_off,
                                            const int *s_prefix, int total0) {
    Tile t;
    if (tile < total0) {
        // last group whose prefix is <= tile
        int lo = 0, hi = p.G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_prefix[mid] <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int g = lo;
        const int cnt = s_off[g + 1] - s_off[g];
        const int mt = (cnt + BM - 1) / BM;
        const int local = tile - s_prefix[g];
        // Keep the larger operand stationary: m fastest when the group's rows
        // are fewer than its weight slice (weights reused from L2 across
        // m-blocks), n fastest otherwise (the A rows reused across n-blocks).
        const bool nfast = cnt > p.brows0;
        const int m_blk = nfast ? local / p.nt0 : local % mt;
        t.seg = 0;
        t.g = g;
        t.row0 = s_off[g] + m_blk * BM;
        t.row_end = s_off[g + 1];
        t.n_blk = nfast ? local % p.nt0 : local / mt;
        t.kblocks = p.K0 / BK;
    } else {
        const int local = tile - total0;
        const int mt = (p.rows1 + BM - 1) / BM;
        const bool nfast = p.rows1 > p.brows1;
        t.seg = 1;
        t.g = 0;
        t.row0 = (nfast ? local / p.nt1 : local % mt) * BM;
        t.row_end = p.rows1;
        t.n_blk = nfast ? local % p.nt1 : local / mt;
        t.kblocks = p.K1 / BK;
    }
    return t;
}

template <int MODE, int BN>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_kernel(const __grid_constant__ Params p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    volatile int *s_bad = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 8);
    int *s_off = reinterpret_cast<int *>(smem + C::OFFS_OFF);
    int *s_prefix = reinterpret_cast<int *>(smem + C::PREFIX_OFF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- prologue: group offsets, tile prefix, barriers
    if (tid == 0) {
        *s_abort = 0;
        *s_bad = 0;
    }
    for (int g = tid; g <= p.G; g += THREADS) s_off[g] = p.offsets[g];
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        bool bad = false;
        for (int g0 = 0; g0 < p.G; g0 += 32) {
            const int g = g0 + lane;
            int tiles = 0;
            if (g < p.G) {
                const int a = s_off[g], b = s_off[g + 1];
                if (a < 0 || b < a || b > p.rows0) bad = true;
                tiles = b > a ? ((b - a + BM - 1) / BM) * p.nt0 : 0;
            }
            int inc = tiles;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += o;
            }
            if (g < p.G) s_prefix[g] = run + inc - tiles;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_prefix[p.G] = run;
        if (__any_sync(0xffffffffu, bad) && lane == 0) *s_bad = 1;
    }
    if (tid == 32) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (*s_bad) {
        if (tid == 0 && blockIdx.x == 0) report(p.dev_status, MOE_DEV_BAD_OFFSETS);
        return;
    }
    const int total0 = s_prefix[p.G];
    const int total = total0 + (p.rows1 > 0 ? ((p.rows1 + BM - 1) / BM) * p.nt1 : 0);

    if (warp == 1) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    if (warp == 0) {
        // ================= TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tmA0);
            tma_prefetch_desc(&p.tmB0);
            if (p.rows1 > 0) {
                tma_prefetch_desc(&p.tmA1);
                tma_prefetch_desc(&p.tmB1);
            }
            int stage = 0;
            uint32_t phase = 0;
            int armed[STAGES];
            for (int s = 0; s < STAGES; ++s) armed[s] = -1;
            for (int tile = blockIdx.x; tile < total && !*s_abort; tile += gridDim.x) {
                const Tile t = decode_tile(p, tile, s_off, s_prefix, total0);
                bool ok = true;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, s_abort, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    armed[stage] = static_cast<int>(phase);
                    uint8_t *a_dst = smem + stage * C::STAGE_BYTES;
                    uint8_t *b_dst = a_dst + A_BYTES;
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    const int k0 = kb * BK;
                    if (t.seg == 0) {
                        tma_load_2d(a_dst, &p.tmA0, &full[stage], k0, t.row0);
                        if (MODE == MODE_SWIGLU) {
                            tma_load_3d(b_dst, &p.tmB0, &full[stage], k0, t.n_blk * 128, t.g);
                            tma_load_3d(b_dst + 128 * BK * 2, &p.tmB0, &full[stage], k0,
                                        p.half0 + t.n_blk * 128, t.g);
                        } else {
                            tma_load_3d(b_dst, &p.tmB0, &full[stage], k0, t.n_blk * BN, t.g);
                        }
                    } else {
                        tma_load_2d(a_dst, &p.tmA1, &full[stage], k0, t.row0);
                        if (MODE == MODE_SWIGLU) {
                            tma_load_2d(b_dst, &p.tmB1, &full[stage], k0, t.n_blk * 128);
                            tma_load_2d(b_dst + 128 * BK * 2, &p.tmB1, &full[stage], k0,
                                        p.half1 + t.n_blk * 128);
                        } else {
                            tma_load_2d(b_dst, &p.tmB1, &full[stage], k0, t.n_blk * BN);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
            }
            if (*s_abort) {
                for (int s = 0; s < STAGES; ++s)
                    if (armed[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(armed[s]));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued = false;
            for (int tile = blockIdx.x; tile < total && !*s_abort; tile += gridDim.x) {
                const Tile t = decode_tile(p, tile, s_off, s_prefix, total0);
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, s_abort, p.dev_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                bool ok = true;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, s_abort, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_bf16(d_tmem, sdesc_kmajor_sw128(a_addr + kk * 32),
                                    sdesc_kmajor_sw128(b_addr + kk * 32), IDESC,
                                    (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            if (*s_abort && issued) {
                // unwinding: wait for every MMA issued so far before TMEM is freed
                tc_commit(drain);
                mbar_wait_drain(drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5)
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int row_in_tile = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode_tile(p, tile, s_off, s_prefix, total0);
            if (!mbar_wait_bounded(&tfull[acc], acc_phase, s_abort, p.dev_status)) break;
            tc_fence_after();
            const int row = t.row0 + row_in_tile;
            const bool ok = row < t.row_end;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            if (MODE == MODE_SWIGLU) {
                uint16_t *out = static_cast<uint16_t *>(t.seg == 0 ? p.out0 : p.out1);
                const int64_t ldo = t.seg == 0 ? p.ldo0 : p.ldo1;
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    float g[32], u[32];
                    __syncwarp();
                    tmem_ld32(taddr + c, g);
                    tmem_ld32(taddr + 128 + c, u);
                    tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float a0 = __fdividef(g[2 * i], 1.0f + __expf(-g[2 * i])) * u[2 * i];
                        const float a1 =
                            __fdividef(g[2 * i + 1], 1.0f + __expf(-g[2 * i + 1])) * u[2 * i + 1];
                        pk[i] = pack_bf16x2(a0, a1);
                    }
                    if (ok) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            out + static_cast<int64_t>(row) * ldo + t.n_blk * 128 + c);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                                                pk[4 * v + 3]);
                    }
                }
            } else {
                const bool f32 = (t.seg == 0 ? p.out0_f32 : p.out1_f32) != 0;
                void *outp = t.seg == 0 ? p.out0 : p.out1;
                const int64_t ldo = t.seg == 0 ? p.ldo0 : p.ldo1;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    __syncwarp();
                    tmem_ld32(taddr + c, v);
                    tmem_ld_wait();
                    if (!ok) continue;
                    const int64_t off = static_cast<int64_t>(row) * ldo + t.n_blk * BN + c;
                    if (f32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(outp) + off);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    } else {
                        uint4 *dst =
                            reinterpret_cast<uint4 *>(static_cast<uint16_t *>(outp) + off);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                                pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                                pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                                pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                    }
                }
            }
            __syncwarp();
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA-pair kernel
// Same tile list and epilogues, but each tile is 256 rows computed by a
// cluster of two CTAs on a TPC with tcgen05.mma.cta_group::2 (M=256, N=256):
// every CTA stages only its own 128 A rows and half of the B slice (32 KB a
// stage instead of 48 KB), so a 6-deep ring fits and the L2 -> shared memory
// traffic per flop drops by a third.
//   - both CTAs' TMA loads complete on the even CTA's full barrier;
//   - one thread of the even CTA issues the MMAs; its commits are multicast
//     to both CTAs (stage release, accumulator ready);
//   - each CTA's epilogue reads its own TMEM rows and arrives on the even
//     CTA's accumulator-empty barrier.
// Tiles are handed out dynamically, in order, from a counter in global
// memory, so the tiles in flight stay a tight window of the list (a static
// round-robin lets lagging clusters drift onto data that has left L2).  The
// even CTA's producer claims each tile and publishes it through a QD-deep
// queue in shared memory: it writes the index into both CTAs' queue slot and
// arrives on both slots' full barriers; the 10 readers (even CTA: MMA thread
// and 4 epilogue warps; odd CTA: producer and 4 epilogue warps) arrive on
// the even CTA's empty barrier once they have read it.  An index >= the
// tile count ends every role's loop.
constexpr int BM2 = 256;
// A stage holds two 64-wide k-slices of A and of B (4 TMA boxes, 64 KB per
// CTA): the producer's per-stage round trip (wait for the slot, arm the
// barrier, issue) limits how fast TMA fills shared memory, and measured on
// GB300 one 64 KB stage streams ~120 GB/s per SM against ~100 GB/s for two
// 32 KB stages (and ~74 GB/s for 16 KB stages).
constexpr int KSUB2 = 2;                      // 64-wide k-slices per stage
constexpr int STAGES2 = 3;
constexpr int STAGE2_BYTES = KSUB2 * 2 * A_BYTES;   // per CTA: KSUB2 x (128x64 A + 128x64 B)
constexpr int TMEM2_COLS = 512;
constexpr int QD = 4;                        // tile-queue depth
constexpr int Q_CONSUMERS = 10;              // see the queue protocol below
constexpr int EPI_BYTES = 32 * 64;           // one 32-row x 64-byte output box

struct Cfg2 {
    static constexpr int EPI_OFF = STAGES2 * STAGE2_BYTES;   // 4 warps x 2 boxes, 1 KB aligned
    static constexpr int BAR_OFF = EPI_OFF + 4 * 2 * EPI_BYTES;
    static constexpr int NBARS = 2 * STAGES2 + 5 + 2 * QD;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int QT_OFF = MISC_OFF + 16;
    static constexpr int OFFS_OFF = QT_OFF + QD * 4;
    static constexpr int PREFIX_OFF = OFFS_OFF + (MAX_GROUPS + 1) * 4;
    static constexpr int SMEM = 1024 + PREFIX_OFF + (MAX_GROUPS + 2) * 4;
};

__device__ __forceinline__ Tile decode_tile_pair(const Params &p, int tile, const int *s_off,
                                                 const int *s_prefix, int total0,
                                                 int ksub = KSUB2) {
    Tile t;
    if (tile < total0) {
        int lo = 0, hi = p.G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_prefix[mid] <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int g = lo;
        const int cnt = s_off[g + 1] - s_off[g];
        const int mt = (cnt + BM2 - 1) / BM2;
        const int local = tile - s_prefix[g];
        const bool nfast = cnt > p.brows0;
        const int m_blk = nfast ? local / p.nt0 : local % mt;
        t.seg = 0;
        t.g = g;
        t.row0 = s_off[g] + m_blk * BM2;
        t.row_end = s_off[g + 1];
        t.n_blk = nfast ? local % p.nt0 : local / mt;
        t.kblocks = p.K0 / (BK * ksub);
    } else {
        const int local = tile - total0;
        const int mt = (p.rows1 + BM2 - 1) / BM2;
        const bool nfast = p.rows1 > p.brows1;
        t.seg = 1;
        t.g = 0;
        t.row0 = (nfast ? local / p.nt1 : local % mt) * BM2;
        t.row_end = p.rows1;
        t.n_blk = nfast ? local % p.nt1 : local / mt;
        t.kblocks = p.K1 / (BK * ksub);
    }
    t.half = t.row_end - t.row0 <= 128;
    return t;
}

// One 32-row x 64-byte output box of an epilogue warp (lane i holds row
// row0 + i as 16 words: 32 bf16 or 16 fp32 values starting at column col).
// The rows are staged in one of the warp's NBOX 2 KB shared-memory boxes in
// the 64-byte swizzle of the output tensor map (16-byte chunk c of row r at
// chunk c ^ ((r >> 1) & 3), conflict-free for the lanes' writes), then leave
// as one TMA tensor store issued by lane 0.  With two boxes the next box is
// written while the store reads the last; with one, the warp first waits for
// the previous store to have read it.
template <int NBOX>
__device__ __forceinline__ void emit_out_box(uint8_t *ebox, int &eb, int lane,
                                             const uint32_t (&w)[16], const CUtensorMap *map,
                                             int col, int row0) {
    static_assert(NBOX == 1 || NBOX == 2, "one or two staging boxes");
    uint8_t *box = ebox + eb * EPI_BYTES;
    if (lane == 0) bulk_wait_read<NBOX - 1>();   // the store that last used this box has read it
    __syncwarp();
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(box + lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(map, box, col, row0);
        bulk_commit();
    }
    if (NBOX == 2) eb ^= 1;
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ Params p) {
    constexpr int BN = 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg2::BAR_OFF);
    uint64_t *full = bars;                      // used in the even CTA only
    uint64_t *empty = bars + STAGES2;
    uint64_t *tfull = bars + 2 * STAGES2;
    uint64_t *tempty = tfull + 2;               // used in the even CTA only
    uint64_t *drain = tempty + 2;
    uint64_t *q_full = drain + 1;               // [QD]
    uint64_t *q_empty = q_full + QD;            // [QD], used in the even CTA only
    volatile int *q_tile = reinterpret_cast<volatile int *>(smem + Cfg2::QT_OFF);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + Cfg2::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + Cfg2::MISC_OFF + 4);
    volatile int *s_bad = reinterpret_cast<volatile int *>(smem + Cfg2::MISC_OFF + 8);
    int *s_off = reinterpret_cast<int *>(smem + Cfg2::OFFS_OFF);
    int *s_prefix = reinterpret_cast<int *>(smem + Cfg2::PREFIX_OFF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();     // 0 = even CTA (issues the MMAs)
    const bool leader = rank == 0;
    const int cid = static_cast<int>(cluster_id_x());

    if (tid == 0) {
        *s_abort = 0;
        *s_bad = 0;
    }
    for (int g = tid; g <= p.G; g += THREADS) s_off[g] = p.offsets[g];
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        bool bad = false;
        for (int g0 = 0; g0 < p.G; g0 += 32) {
            const int g = g0 + lane;
            int tiles = 0;
            if (g < p.G) {
                const int a = s_off[g], b = s_off[g + 1];
                if (a < 0 || b < a || b > p.rows0) bad = true;
                tiles = b > a ? ((b - a + BM2 - 1) / BM2) * p.nt0 : 0;
            }
            int inc = tiles;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += o;
            }
            if (g < p.G) s_prefix[g] = run + inc - tiles;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_prefix[p.G] = run;
        if (__any_sync(0xffffffffu, bad) && lane == 0) *s_bad = 1;
    }
    if (tid == 32) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);    // lane 0 of the 4 epilogue warps of both CTAs
        }
        mbar_init(drain, 1);
        for (int q = 0; q < QD; ++q) {
            mbar_init(&q_full[q], 1);
            mbar_init(&q_empty[q], Q_CONSUMERS);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // both CTAs read the same offsets, so both leave here together
    if (*s_bad) {
        if (tid == 0 && cid == 0 && leader) report(p.dev_status, MOE_DEV_BAD_OFFSETS);
        return;
    }
    const int total0 = s_prefix[p.G];
    const int total = total0 + (p.rows1 > 0 ? ((p.rows1 + BM2 - 1) / BM2) * p.nt1 : 0);

    if (warp == 1) {
        tmem_alloc_pair(s_tmem, TMEM2_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();          // barriers and TMEM of both CTAs are ready
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const uint32_t lead_full = mapa_shared(smem_u32(full), 0);
    const uint32_t lead_tempty = mapa_shared(smem_u32(tempty), 0);
    const uint32_t lead_qempty = mapa_shared(smem_u32(q_empty), 0);
    const uint32_t peer_qfull = mapa_shared(smem_u32(q_full), 1);
    const uint32_t peer_qtile = mapa_shared(static_cast<uint32_t>(__cvta_generic_to_shared(
                                                const_cast<int *>(q_tile))), 1);
    // Reader side of the tile queue (all roles but the even CTA's producer).
    // Returns false when a wait gave up.
    auto next_tile = [&](int &qi, uint32_t &qph, int &tile) -> bool {
        if (!mbar_wait_bounded_cluster(&q_full[qi], qph, s_abort, p.dev_status)) return false;
        tile = q_tile[qi];
        mbar_arrive_cluster(lead_qempty + 8u * static_cast<uint32_t>(qi));
        if (++qi == QD) {
            qi = 0;
            qph ^= 1;
        }
        return true;
    };

    if (warp == 0) {
        // ================= TMA producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&p.tmA0);
            tma_prefetch_desc(&p.tmB0);
            if (p.rows1 > 0) {
                tma_prefetch_desc(&p.tmA1);
                tma_prefetch_desc(&p.tmB1);
            }
            int stage = 0;
            uint32_t phase = 0;
            int armed[STAGES2];
            for (int s = 0; s < STAGES2; ++s) armed[s] = -1;
            int qi = 0;
            uint32_t qph = 0;
            while (!*s_abort) {
                int tile;
                if (leader) {
                    // claim the next tile and publish it to both CTAs
                    if (!mbar_wait_bounded_cluster(&q_empty[qi], qph ^ 1, s_abort, p.dev_status))
                        break;
                    tile = static_cast<int>(atomicAdd(p.tile_counter, 1u));
                    q_tile[qi] = tile;
                    mbar_arrive(&q_full[qi]);
                    st_shared_cluster_u32(peer_qtile + 4u * static_cast<uint32_t>(qi),
                                          static_cast<uint32_t>(tile));
                    mbar_arrive_cluster(peer_qfull + 8u * static_cast<uint32_t>(qi));
                    if (++qi == QD) {
                        qi = 0;
                        qph ^= 1;
                    }
                } else if (!next_tile(qi, qph, tile)) {
                    break;
                }
                if (tile >= total) break;
                const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0);
                // a half tile (M=128) takes 64 rows per CTA
                const int arow = t.row0 + (t.half ? 64 : 128) * static_cast<int>(rank);
                const uint32_t stage_tx =
                    t.half ? 2u * KSUB2 * (A_BYTES / 2 + A_BYTES) : 2u * STAGE2_BYTES;
                bool ok = true;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, s_abort, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    armed[stage] = static_cast<int>(phase);
                    uint8_t *a_dst = smem + stage * STAGE2_BYTES;
                    uint8_t *b_dst = a_dst + KSUB2 * A_BYTES;
                    if (leader) mbar_arrive_expect_tx(&full[stage], stage_tx);
                    const uint32_t fb = lead_full + 8u * static_cast<uint32_t>(stage);
                    const int whalf = t.seg == 0 ? p.half0 : p.half1;
                    int brow;
                    if (MODE == MODE_SWIGLU)
                        brow = (rank == 0 ? 0 : whalf) + t.n_blk * 128;
                    else
                        brow = t.n_blk * BN + 128 * static_cast<int>(rank);
#pragma unroll
                    for (int sub = 0; sub < KSUB2; ++sub) {
                        const int k0 = (kb * KSUB2 + sub) * BK;
                        uint8_t *ad = a_dst + sub * A_BYTES;
                        uint8_t *bd = b_dst + sub * A_BYTES;
                        if (!t.half) {
                            if (t.seg == 0) {
                                tma_load_2d_pair(ad, &p.tmA0, fb, k0, arow);
                                tma_load_3d_pair(bd, &p.tmB0, fb, k0, brow, t.g);
                            } else {
                                tma_load_2d_pair(ad, &p.tmA1, fb, k0, arow);
                                tma_load_2d_pair(bd, &p.tmB1, fb, k0, brow);
                            }
                        } else if (MODE == MODE_SWIGLU) {
                            // this CTA's half of B: 64 gate rows then the 64 matching up rows
                            const int grow = t.n_blk * 128 + 64 * static_cast<int>(rank);
                            if (t.seg == 0) {
                                tma_load_2d_pair(ad, &p.tmA0h, fb, k0, arow);
                                tma_load_3d_pair(bd, &p.tmB0h, fb, k0, grow, t.g);
                                tma_load_3d_pair(bd + A_BYTES / 2, &p.tmB0h, fb, k0, whalf + grow,
                                                 t.g);
                            } else {
                                tma_load_2d_pair(ad, &p.tmA1h, fb, k0, arow);
                                tma_load_2d_pair(bd, &p.tmB1h, fb, k0, grow);
                                tma_load_2d_pair(bd + A_BYTES / 2, &p.tmB1h, fb, k0, whalf + grow);
                            }
                        } else {
                            if (t.seg == 0) {
                                tma_load_2d_pair(ad, &p.tmA0h, fb, k0, arow);
                                tma_load_3d_pair(bd, &p.tmB0, fb, k0, brow, t.g);
                            } else {
                                tma_load_2d_pair(ad, &p.tmA1h, fb, k0, arow);
                                tma_load_2d_pair(bd, &p.tmB1, fb, k0, brow);
                            }
                        }
                    }
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
            }
            if (*s_abort && leader) {
                for (int s = 0; s < STAGES2; ++s)
                    if (armed[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(armed[s]));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (even CTA only)
        if (lane == 0 && leader) {
            constexpr uint32_t IDESC = idesc_bf16_f32(BM2, BN);
            // M=128 over the pair (64 rows per CTA) takes half the MMA time;
            // its accumulator occupies 128 columns: rows in lanes 0-63 with
            // columns 0-127 of N, the same rows again in lanes 64-127 with
            // columns 128-255 (measured on GB300)
            constexpr uint32_t IDESC_HALF = idesc_bf16_f32(BM2 / 2, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued = false;
            int qi = 0;
            uint32_t qph = 0;
            while (!*s_abort) {
                int tile;
                if (!next_tile(qi, qph, tile) || tile >= total) break;
                const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0);
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, s_abort, p.dev_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                bool ok = true;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, s_abort, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * STAGE2_BYTES);
                    const uint32_t b_addr = a_addr + KSUB2 * A_BYTES;
#pragma unroll
                    for (int sub = 0; sub < KSUB2; ++sub)
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint32_t off = sub * A_BYTES + kk * 32;
                            tc_mma_bf16_pair(d_tmem, sdesc_kmajor_sw128(a_addr + off),
                                             sdesc_kmajor_sw128(b_addr + off), t.half ? IDESC_HALF : IDESC,
                                             (kb | sub | kk) != 0 ? 1u : 0u);
                        }
                    issued = true;
                    tc_commit_pair_mc(&empty[stage], 0x3);
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc(&tfull[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            if (*s_abort && issued) {
                tc_commit_pair_mc(drain, 0x1);
                mbar_wait_drain(drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5 of both CTAs)
        const int q = warp & 3;
        const int row_in_tile = 128 * static_cast<int>(rank) + q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        int qi = 0;
        uint32_t qph = 0;
        // Two 2 KB staging boxes per warp.  A box holds 32 rows x 64 bytes in
        // the 64-byte swizzle of the output tensor map (16-byte chunk c of
        // row r sits at chunk c ^ ((r >> 1) & 3)), which also keeps the
        // lanes' shared-memory writes free of bank conflicts.
        uint8_t *ebox = smem + Cfg2::EPI_OFF + (warp - 2) * 2 * EPI_BYTES;
        int eb = 0;
        auto emit_box = [&](const uint32_t(&w)[16], const CUtensorMap *map, int col, int row0) {
            emit_out_box<2>(ebox, eb, lane, w, map, col, row0);
        };
        for (;;) {
            int tile = 0, got = 1;
            if (lane == 0) {
                // one reader per warp: wait, read, release the slot
                if (mbar_wait_bounded_cluster(&q_full[qi], qph, s_abort, p.dev_status)) {
                    tile = q_tile[qi];
                    mbar_arrive_cluster(lead_qempty + 8u * static_cast<uint32_t>(qi));
                } else {
                    got = 0;
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (++qi == QD) {
                qi = 0;
                qph ^= 1;
            }
            if (!got || tile >= total) break;
            const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0);
            if (!mbar_wait_bounded(&tfull[acc], acc_phase, s_abort, p.dev_status)) break;
            tc_fence_after();
            // full tile: this CTA's 128 rows, warp quadrant q = rows 32q..;
            // half tile: this CTA's 64 rows, quadrant q = rows 32(q & 1).. of
            // the columns' half q >> 1 (see the MMA's TMEM layout)
            const int hq = q >> 1;
            const int row = t.half ? t.row0 + 64 * static_cast<int>(rank) + 32 * (q & 1) + lane
                                   : t.row0 + row_in_tile;
            const bool ok = row < t.row_end;
            // All 32 rows of this warp inside the group: the results leave
            // through TMA stores of whole 32-row boxes; otherwise (a group's
            // last block) each lane stores its own row if it is in range.
            const int row_base = row - lane;
            const bool boxed = row_base + 32 <= t.row_end;
            const CUtensorMap *omap = t.seg == 0 ? &p.tmO0 : &p.tmO1;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            if (MODE == MODE_SWIGLU) {
                uint16_t *out = static_cast<uint16_t *>(t.seg == 0 ? p.out0 : p.out1);
                const int64_t ldo = t.seg == 0 ? p.ldo0 : p.ldo1;
                // gate in columns [0, w), up in [w, 2w): w = 128 (full) or 64 (half)
                const int uoff = t.half ? 64 : 128;
                const int col0 = t.n_blk * 128 + (t.half ? 64 * hq : 0);
#pragma unroll 1
                for (int c = 0; c < uoff; c += 32) {
                    float g[32], u[32];
                    __syncwarp();
                    tmem_ld32(taddr + c, g);
                    tmem_ld32(taddr + uoff + c, u);
                    tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float a0 = __fdividef(g[2 * i], 1.0f + __expf(-g[2 * i])) * u[2 * i];
                        const float a1 =
                            __fdividef(g[2 * i + 1], 1.0f + __expf(-g[2 * i + 1])) * u[2 * i + 1];
                        pk[i] = pack_bf16x2(a0, a1);
                    }
                    if (boxed) {
                        emit_box(pk, omap, col0 + c, row_base);
                    } else if (ok) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            out + static_cast<int64_t>(row) * ldo + col0 + c);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                                                pk[4 * v + 3]);
                    }
                }
            } else {
                const bool f32 = (t.seg == 0 ? p.out0_f32 : p.out1_f32) != 0;
                void *outp = t.seg == 0 ? p.out0 : p.out1;
                const int64_t ldo = t.seg == 0 ? p.ldo0 : p.ldo1;
                const int ncol = t.half ? BN / 2 : BN;
                const int col0 = t.n_blk * BN + (t.half ? (BN / 2) * hq : 0);
#pragma unroll 1
                for (int c = 0; c < ncol; c += 32) {
                    float v[32];
                    __syncwarp();
                    tmem_ld32(taddr + c, v);
                    tmem_ld_wait();
                    const int col = col0 + c;
                    if (boxed) {
                        if (f32) {
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i]);
                            emit_box(w, omap, col, row_base);
#pragma unroll
                            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[16 + i]);
                            emit_box(w, omap, col + 16, row_base);
                        } else {
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                            emit_box(w, omap, col, row_base);
                        }
                        continue;
                    }
                    if (!ok) continue;
                    const int64_t off = static_cast<int64_t>(row) * ldo + col;
                    if (f32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(outp) + off);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    } else {
                        uint4 *dst =
                            reinterpret_cast<uint4 *>(static_cast<uint16_t *>(outp) + off);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                                pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                                pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                                pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                    }
                }
            }
            __syncwarp();
            tc_fence_before();
            if (lane == 0) mbar_arrive_cluster(lead_tempty + 8u * static_cast<uint32_t>(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        if (lane == 0) bulk_wait<0>();   // every output box written
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();          // no CTA leaves while its peer may still signal or read it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM2_COLS);
    }
}

// ------------------------------------------------------------------ wide CTA-pair kernel
// Tiles of 256 rows x 512 accumulator columns per CTA pair: per 64-wide
// k-slice each CTA stages its 128 A rows (16 KB) and 256 rows of B (32 KB),
// and the MMA thread issues two M=256, N=256 pair MMAs (accumulator halves
// 0 and 1, TMEM columns [0, 256) and [256, 512)).  Per flop that is a
// quarter fewer bytes through the SM's TMA engine than the 256 x 256 pair
// tiles (48 KB for 2 x 256 x 512 x 64 flops against 32 KB for half that),
// which is the limit of the operand fill when the clock is not capped.
//   SWIGLU: the tile covers 256 act columns; the even CTA stages the 256
//     gate rows, the odd CTA the matching 256 up rows, so half h holds g in
//     its columns [0, 128) and u in [128, 256) for act columns 128h + j.
//   STORE: the tile covers 512 output columns; CTA r stages B rows
//     [256r, 256r + 256), so TMEM column 256h + j holds output column
//     128h + j (j < 128) or 256 + 128h + (j - 128) (j >= 128).
// The single 512-column accumulator is not double-buffered.  Instead eight
// epilogue warps per CTA (two per TMEM lane quarter) drain half 0 first and
// release it, then half 1; the MMA thread starts the next tile on half 0 as
// soon as that is free and runs ahead on it over the staged k-slices (their
// stages are released only once the half-1 MMAs of the slice are issued)
// until half 1 is free too.  A four-deep ring of 48 KB stages gives that
// run-ahead room and leaves shared memory for one staging box per warp: the
// output leaves as TMA tensor stores, each warp waiting for its previous
// store to have read the box (measured against the same box read back and
// written through the load/store units: the down matmul 1.8-3.6% faster).
// A group's last block of at most 128 rows runs as M=128 pair MMAs (64 rows
// per CTA): MMA h then occupies TMEM columns [256h, 256h + 128), the CTA's
// 64 rows in lanes 0-63 for N columns 0-127 and again in lanes 64-127 for
// N columns 128-255; in SWIGLU mode each CTA then stages, per half, 64 gate
// rows and the matching 64 up rows.
// Tile queue, bounded waits and unwinding as in the pair kernel above.
constexpr int WSTAGES = 4;
constexpr int W_BOXES = 1;                              // staging box per epilogue warp
constexpr int W_B_BYTES = 2 * A_BYTES;                  // 256 rows x 64 bf16
constexpr int W_STAGE_BYTES = A_BYTES + W_B_BYTES;      // 48 KB per CTA
constexpr int W_EPI_WARPS = 8;
constexpr int W_THREADS = 64 + 32 * W_EPI_WARPS;
constexpr int WQ_CONSUMERS = 2 + 2 * W_EPI_WARPS;       // MMA thread, odd producer, epilogue
// With gathered A, four more warps per CTA copy each stage's A rows (16-byte
// cp.async, straight into the 128-byte swizzle), and the odd CTA's warp 1
// relays "A landed" to the even CTA's full barrier.
// The last W_TAIL k-blocks of a tile issue their half-1 MMAs after all
// half-0 ones: half 0 is reported complete that much earlier and the
// epilogue drains it while they run.  Measured on T=16384, H=4096, I=3072:
// both matmuls ~1% faster with 3 than with none; with 4 (the whole ring
// held back) the gain is gone.
constexpr int W_TAIL = 3;
constexpr int W_GATHER_WARPS = 4;
constexpr int W_THREADS_G = W_THREADS + 32 * W_GATHER_WARPS;
constexpr int WQ_CONSUMERS_G = WQ_CONSUMERS + 2 * W_GATHER_WARPS + 1;
struct CfgW {
    static constexpr int EPI_OFF = WSTAGES * W_STAGE_BYTES;
    static constexpr int BAR_OFF = EPI_OFF + W_EPI_WARPS * W_BOXES * EPI_BYTES;
    // full[S], empty[S], tfull[2], tempty[2], drain, q_full[QD], q_empty[QD], a_full[S]
    static constexpr int NBARS = 3 * WSTAGES + 5 + 2 * QD;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int QT_OFF = MISC_OFF + 16;
    static constexpr int OFFS_OFF = QT_OFF + QD * 4;
    static constexpr int PREFIX_OFF = OFFS_OFF + (MAX_GROUPS + 1) * 4;
    static constexpr int SMEM = 1024 + PREFIX_OFF + (MAX_GROUPS + 2) * 4;
};
static_assert(CfgW::SMEM <= 227 * 1024, "wide pair kernel: shared memory");


template <int MODE, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GATHER ? W_THREADS_G : W_THREADS, 1)
    grouped_gemm_wide_kernel(const __grid_constant__ Params p) {
    constexpr int NT = GATHER ? W_THREADS_G : W_THREADS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + CfgW::BAR_OFF);
    uint64_t *full = bars;                      // used in the even CTA only
    uint64_t *empty = bars + WSTAGES;
    uint64_t *tfull = bars + 2 * WSTAGES;       // [2]: accumulator half h complete
    uint64_t *tempty = tfull + 2;               // [2], used in the even CTA only
    uint64_t *drain = tempty + 2;
    uint64_t *q_full = drain + 1;               // [QD]
    uint64_t *q_empty = q_full + QD;            // [QD], used in the even CTA only
    uint64_t *a_full = q_empty + QD;            // [WSTAGES]: this CTA's gathered A landed
    volatile int *q_tile = reinterpret_cast<volatile int *>(smem + CfgW::QT_OFF);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + CfgW::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + CfgW::MISC_OFF + 4);
    volatile int *s_bad = reinterpret_cast<volatile int *>(smem + CfgW::MISC_OFF + 8);
    int *s_off = reinterpret_cast<int *>(smem + CfgW::OFFS_OFF);
    int *s_prefix = reinterpret_cast<int *>(smem + CfgW::PREFIX_OFF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cid = static_cast<int>(cluster_id_x());

    if (tid == 0) {
        *s_abort = 0;
        *s_bad = 0;
    }
    for (int g = tid; g <= p.G; g += NT) s_off[g] = p.offsets[g];
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        bool bad = false;
        for (int g0 = 0; g0 < p.G; g0 += 32) {
            const int g = g0 + lane;
            int tiles = 0;
            if (g < p.G) {
                const int a = s_off[g], b = s_off[g + 1];
                if (a < 0 || b < a || b > p.rows0) bad = true;
                tiles = b > a ? ((b - a + BM2 - 1) / BM2) * p.nt0 : 0;
            }
            int inc = tiles;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += o;
            }
            if (g < p.G) s_prefix[g] = run + inc - tiles;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_prefix[p.G] = run;
        if (__any_sync(0xffffffffu, bad) && lane == 0) *s_bad = 1;
    }
    if (tid == 32) {
        for (int s = 0; s < WSTAGES; ++s) {
            // even CTA: its producer's arming arrival (+ the odd CTA's relay of
            // its gathered A)
            mbar_init(&full[s], GATHER ? 2 : 1);
            mbar_init(&empty[s], 1);
            mbar_init(&a_full[s], 32 * W_GATHER_WARPS);
        }
        mbar_init(&tfull[0], 1);
        mbar_init(&tfull[1], 1);
        mbar_init(&tempty[0], 2 * W_EPI_WARPS);   // lane 0 of every epilogue warp of both CTAs
        mbar_init(&tempty[1], 2 * W_EPI_WARPS);
        mbar_init(drain, 1);
        for (int q = 0; q < QD; ++q) {
            mbar_init(&q_full[q], 1);
            mbar_init(&q_empty[q], GATHER ? WQ_CONSUMERS_G : WQ_CONSUMERS);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (*s_bad) {
        if (tid == 0 && cid == 0 && leader) report(p.dev_status, MOE_DEV_BAD_OFFSETS);
        return;
    }
    const int total0 = s_prefix[p.G];
    const int total = total0 + (p.rows1 > 0 ? ((p.rows1 + BM2 - 1) / BM2) * p.nt1 : 0);

    if (warp == 1) {
        tmem_alloc_pair(s_tmem, TMEM2_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const uint32_t lead_full = mapa_shared(smem_u32(full), 0);
    const uint32_t lead_tempty = mapa_shared(smem_u32(tempty), 0);
    const uint32_t lead_qempty = mapa_shared(smem_u32(q_empty), 0);
    const uint32_t peer_qfull = mapa_shared(smem_u32(q_full), 1);
    const uint32_t peer_qtile = mapa_shared(static_cast<uint32_t>(__cvta_generic_to_shared(
                                                const_cast<int *>(q_tile))), 1);
    auto next_tile = [&](int &qi, uint32_t &qph, int &tile) -> bool {
        if (!mbar_wait_bounded_cluster(&q_full[qi], qph, s_abort, p.dev_status)) return false;
        tile = q_tile[qi];
        mbar_arrive_cluster(lead_qempty + 8u * static_cast<uint32_t>(qi));
        if (++qi == QD) {
            qi = 0;
            qph ^= 1;
        }
        return true;
    };

    if (warp == 0) {
        // ================= TMA producer (both CTAs)
        if (lane == 0) {
            if (!GATHER) tma_prefetch_desc(&p.tmA0);
            tma_prefetch_desc(&p.tmB0w);
            if (p.rows1 > 0) {
                if (!GATHER) tma_prefetch_desc(&p.tmA1);
                tma_prefetch_desc(&p.tmB1w);
            }
            int stage = 0;
            uint32_t phase = 0;
            int armed[WSTAGES];
            for (int s = 0; s < WSTAGES; ++s) armed[s] = -1;
            int qi = 0;
            uint32_t qph = 0;
            while (!*s_abort) {
                int tile;
                if (leader) {
                    if (!mbar_wait_bounded_cluster(&q_empty[qi], qph ^ 1, s_abort, p.dev_status))
                        break;
                    tile = static_cast<int>(atomicAdd(p.tile_counter, 1u));
                    q_tile[qi] = tile;
                    mbar_arrive(&q_full[qi]);
                    st_shared_cluster_u32(peer_qtile + 4u * static_cast<uint32_t>(qi),
                                          static_cast<uint32_t>(tile));
                    mbar_arrive_cluster(peer_qfull + 8u * static_cast<uint32_t>(qi));
                    if (++qi == QD) {
                        qi = 0;
                        qph ^= 1;
                    }
                } else if (!next_tile(qi, qph, tile)) {
                    break;
                }
                if (tile >= total) break;
                const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0, 1);
                const int arow = t.row0 + (t.half ? 64 : 128) * static_cast<int>(rank);
                // bytes of both CTAs (with gathered A: B only)
                const uint32_t stage_tx =
                    GATHER ? 2u * W_B_BYTES
                           : (t.half ? 2u * (A_BYTES / 2 + W_B_BYTES) : 2u * W_STAGE_BYTES);
                const int whalf = t.seg == 0 ? p.half0 : p.half1;
                const CUtensorMap *mA = t.seg == 0 ? (t.half ? &p.tmA0h : &p.tmA0)
                                                   : (t.half ? &p.tmA1h : &p.tmA1);
                const CUtensorMap *mBw = t.seg == 0 ? &p.tmB0w : &p.tmB1w;
                const CUtensorMap *mBh = t.seg == 0 ? &p.tmB0h : &p.tmB1h;
                bool ok = true;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, s_abort, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    armed[stage] = static_cast<int>(phase);
                    uint8_t *a_dst = smem + stage * W_STAGE_BYTES;
                    uint8_t *b_dst = a_dst + A_BYTES;
                    if (leader) mbar_arrive_expect_tx(&full[stage], stage_tx);
                    const uint32_t fb = lead_full + 8u * static_cast<uint32_t>(stage);
                    const int k0 = kb * BK;
                    if (!GATHER) tma_load_2d_pair(a_dst, mA, fb, k0, arow);
                    if (MODE == MODE_SWIGLU && t.half) {
                        // per half: 64 gate rows, then the matching 64 up rows
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int grow = t.n_blk * 256 + 128 * h + 64 * static_cast<int>(rank);
                            uint8_t *bd = b_dst + h * A_BYTES;
                            if (t.seg == 0) {
                                tma_load_3d_pair(bd, mBh, fb, k0, grow, t.g);
                                tma_load_3d_pair(bd + A_BYTES / 2, mBh, fb, k0, whalf + grow, t.g);
                            } else {
                                tma_load_2d_pair(bd, mBh, fb, k0, grow);
                                tma_load_2d_pair(bd + A_BYTES / 2, mBh, fb, k0, whalf + grow);
                            }
                        }
                    } else {
                        const int brow = MODE == MODE_SWIGLU
                                             ? (rank == 0 ? 0 : whalf) + t.n_blk * 256
                                             : t.n_blk * 512 + 256 * static_cast<int>(rank);
                        if (t.seg == 0)
                            tma_load_3d_pair(b_dst, mBw, fb, k0, brow, t.g);
                        else
                            tma_load_2d_pair(b_dst, mBw, fb, k0, brow);
                    }
                    if (++stage == WSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
            }
            if (*s_abort && leader) {
                for (int s = 0; s < WSTAGES; ++s)
                    if (armed[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(armed[s]));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (even CTA only)
        if (lane == 0 && leader) {
            constexpr uint32_t IDESC = idesc_bf16_f32(BM2, 256);
            constexpr uint32_t IDESC_HALF = idesc_bf16_f32(BM2 / 2, 256);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t tph = 0;
            bool issued = false;
            int qi = 0;
            uint32_t qph = 0;
            while (!*s_abort) {
                int tile;
                if (!next_tile(qi, qph, tile) || tile >= total) break;
                const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0, 1);
                const uint32_t idesc = t.half ? IDESC_HALF : IDESC;
                // accumulator half h of stage st, k-block kb
                auto mma_half = [&](int st, int kb, int h) {
                    const uint32_t a_addr = smem_u32(smem + st * W_STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_BYTES + static_cast<uint32_t>(h) * A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_bf16_pair(tmem_base + 256u * static_cast<uint32_t>(h),
                                         sdesc_kmajor_sw128(a_addr + kk * 32),
                                         sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                                         (kb | kk) != 0 ? 1u : 0u);
                };
                if (!mbar_wait_bounded_cluster(&tempty[0], tph ^ 1, s_abort, p.dev_status)) break;
                tc_fence_after();
                bool h1 = false;
                const int tail_from = t.kblocks - min(W_TAIL, t.kblocks);
                int pend_st[WSTAGES];
                int npend = 0, pend_kb0 = 0;
                auto flush = [&]() {
                    for (int i = 0; i < npend; ++i) {
                        mma_half(pend_st[i], pend_kb0 + i, 1);
                        tc_commit_pair_mc(&empty[pend_st[i]], 0x3);
                    }
                    npend = 0;
                };
                bool ok = true;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    // with gathered A: the odd CTA's A arrives through full[] (its
                    // relay), this CTA's through a_full[]
                    const bool got_full =
                        GATHER ? mbar_wait_bounded_cluster(&full[stage], phase, s_abort, p.dev_status)
                               : mbar_wait_bounded(&full[stage], phase, s_abort, p.dev_status);
                    if (!got_full ||
                        (GATHER && !mbar_wait_bounded(&a_full[stage], phase, s_abort, p.dev_status))) {
                        ok = false;
                        break;
                    }
                    // the gathered rows were written through the generic proxy;
                    // the tensor core reads them through the async proxy
                    if (GATHER) fence_proxy_async();
                    tc_fence_after();
                    mma_half(stage, kb, 0);
                    issued = true;
                    // the tile's last k-blocks keep their half-1 MMAs back
                    const bool tail = kb >= tail_from;
                    if (!tail && !h1 && mbar_test_wait_cluster(&tempty[1], tph ^ 1)) {
                        tc_fence_after();
                        h1 = true;
                    }
                    if (h1 && !tail) {
                        flush();
                        mma_half(stage, kb, 1);
                        tc_commit_pair_mc(&empty[stage], 0x3);
                    } else {
                        if (npend == 0) pend_kb0 = kb;
                        pend_st[npend++] = stage;
                        if (npend == WSTAGES) {
                            // every stage waits for half 1: the producer cannot go on
                            if (!h1) {
                                if (!mbar_wait_bounded_cluster(&tempty[1], tph ^ 1, s_abort,
                                                               p.dev_status)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                h1 = true;
                            }
                            flush();
                        }
                    }
                    if (++stage == WSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                // half 0 is complete once every MMA issued so far is: the
                // epilogue drains it while the held-back half-1 MMAs run
                tc_commit_pair_mc(&tfull[0], 0x3);
                if (npend > 0) {
                    if (!h1) {
                        if (!mbar_wait_bounded_cluster(&tempty[1], tph ^ 1, s_abort,
                                                       p.dev_status))
                            break;
                        tc_fence_after();
                        h1 = true;
                    }
                    flush();
                }
                tc_commit_pair_mc(&tfull[1], 0x3);
                tph ^= 1;
            }
            if (*s_abort && issued) {
                tc_commit_pair_mc(drain, 0x1);
                mbar_wait_drain(drain, 0);
            }
        } else if (GATHER && lane == 0 && !leader) {
            // ================= relay (odd CTA): each stage's gathered A rows of
            // this CTA have landed -> arrive on the even CTA's full barrier
            int stage = 0;
            uint32_t phase = 0;
            int qi = 0;
            uint32_t qph = 0;
            while (!*s_abort) {
                int tile;
                if (!next_tile(qi, qph, tile) || tile >= total) break;
                const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0, 1);
                bool ok = true;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait_bounded(&a_full[stage], phase, s_abort, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async();
                    mbar_arrive_cluster(lead_full + 8u * static_cast<uint32_t>(stage));
                    if (++stage == WSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp < W_THREADS / 32) {
        // ================= epilogue (warps 2..9 of both CTAs)
        const int q = warp & 3;            // TMEM lane quarter this warp may read
        const int sub = (warp - 2) >> 2;   // which half of the quarter's columns
        uint32_t tph = 0;
        int qi = 0;
        uint32_t qph = 0;
        uint8_t *ebox = smem + CfgW::EPI_OFF + (warp - 2) * W_BOXES * EPI_BYTES;
        int eb = 0;
        auto emit_box = [&](const uint32_t(&w)[16], const CUtensorMap *map, int col, int row0) {
            emit_out_box<W_BOXES>(ebox, eb, lane, w, map, col, row0);
        };
        for (;;) {
            int tile = 0, got = 1;
            if (lane == 0) {
                if (mbar_wait_bounded_cluster(&q_full[qi], qph, s_abort, p.dev_status)) {
                    tile = q_tile[qi];
                    mbar_arrive_cluster(lead_qempty + 8u * static_cast<uint32_t>(qi));
                } else {
                    got = 0;
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (++qi == QD) {
                qi = 0;
                qph ^= 1;
            }
            if (!got || tile >= total) break;
            const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0, 1);
            const int hq = q >> 1;
            const int row = t.half ? t.row0 + 64 * static_cast<int>(rank) + 32 * (q & 1) + lane
                                   : t.row0 + 128 * static_cast<int>(rank) + 32 * q + lane;
            const bool ok = row < t.row_end;
            const int row_base = row - lane;
            const bool boxed = row_base + 32 <= t.row_end;
            const CUtensorMap *omap = t.seg == 0 ? &p.tmO0 : &p.tmO1;
            const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            bool stop = false;
            for (int h = 0; h < 2; ++h) {
                if (!mbar_wait_bounded(&tfull[h], tph, s_abort, p.dev_status)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                if (MODE == MODE_SWIGLU) {
                    uint16_t *out = static_cast<uint16_t *>(t.seg == 0 ? p.out0 : p.out1);
                    const int64_t ldo = t.seg == 0 ? p.ldo0 : p.ldo1;
                    // full: g at 256h + [0,128), u at 256h + 128 + [0,128), act 128h + j;
                    // half: g at 256h + [0,64), u at 256h + 64 + [0,64), act 128h + 64 hq + j
                    const int uoff = t.half ? 64 : 128;
                    const int ncol = t.half ? 32 : 64;          // this warp's share
                    const int j0 = ncol * sub;
                    const int act0 = t.n_blk * 256 + 128 * h + (t.half ? 64 * hq : 0) + j0;
                    const uint32_t gbase = tq + 256u * static_cast<uint32_t>(h) + j0;
#pragma unroll 1
                    for (int c = 0; c < ncol; c += 32) {
                        uint32_t pk[16];
                        // 16 columns of g and u at a time (fewer live registers)
#pragma unroll
                        for (int hc = 0; hc < 32; hc += 16) {
                            float g[16], u[16];
                            __syncwarp();
                            tmem_ld16(gbase + c + hc, g);
                            tmem_ld16(gbase + uoff + c + hc, u);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float a0 =
                                    __fdividef(g[2 * i], 1.0f + __expf(-g[2 * i])) * u[2 * i];
                                const float a1 =
                                    __fdividef(g[2 * i + 1], 1.0f + __expf(-g[2 * i + 1])) *
                                    u[2 * i + 1];
                                pk[hc / 2 + i] = pack_bf16x2(a0, a1);
                            }
                        }
                        if (boxed) {
                            emit_box(pk, omap, act0 + c, row_base);
                        } else if (ok) {
                            uint4 *dst = reinterpret_cast<uint4 *>(
                                out + static_cast<int64_t>(row) * ldo + act0 + c);
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                                                    pk[4 * v + 3]);
                        }
                    }
                } else {
                    const bool f32 = (t.seg == 0 ? p.out0_f32 : p.out1_f32) != 0;
                    void *outp = t.seg == 0 ? p.out0 : p.out1;
                    const int64_t ldo = t.seg == 0 ? p.ldo0 : p.ldo1;
                    // full: TMEM 256h + 128 sub + [0,128) -> out 256 sub + 128h + j;
                    // half: TMEM 256h + 64 sub + [0,64) -> out 256 hq + 128h + 64 sub + j
                    const int ncol = t.half ? 64 : 128;
                    const uint32_t tbase = tq + 256u * static_cast<uint32_t>(h) + ncol * sub;
                    const int col0 = t.n_blk * 512 + 128 * h +
                                     (t.half ? 256 * hq + 64 * sub : 256 * sub);
#pragma unroll 1
                    for (int c = 0; c < ncol; c += 32) {
                        float v[32];
                        __syncwarp();
                        tmem_ld32(tbase + c, v);
                        tmem_ld_wait();
                        const int col = col0 + c;
                        if (boxed) {
                            uint32_t w[16];
                            if (f32) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i]);
                                emit_box(w, omap, col, row_base);
#pragma unroll
                                for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[16 + i]);
                                emit_box(w, omap, col + 16, row_base);
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                                emit_box(w, omap, col, row_base);
                            }
                            continue;
                        }
                        if (!ok) continue;
                        const int64_t off = static_cast<int64_t>(row) * ldo + col;
                        if (f32) {
                            float4 *dst =
                                reinterpret_cast<float4 *>(static_cast<float *>(outp) + off);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[i] =
                                    make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        } else {
                            uint4 *dst =
                                reinterpret_cast<uint4 *>(static_cast<uint16_t *>(outp) + off);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                                    pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                                    pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                                    pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                        }
                    }
                }
                // this warp's columns of half h have left TMEM
                __syncwarp();
                tc_fence_before();
                if (lane == 0) mbar_arrive_cluster(lead_tempty + 8u * static_cast<uint32_t>(h));
            }
            if (stop) break;
            tph ^= 1;
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    } else if (GATHER) {
        // ================= A gather (warps 10..13 of both CTAs): this CTA's
        // 128 (half tile: 64) A rows of each stage, 16-byte cp.async copies
        // into the 128-byte swizzle (chunk j of row r at (j ^ (r & 7)) * 16),
        // 8 threads per 128-byte row piece.  Each thread's copies of a stage
        // arrive on a_full[stage] by themselves once they have landed, so the
        // gather runs as far ahead as the free slots allow.
        const int gt = tid - W_THREADS;     // 0..127
        const int j = gt & 7;               // 16-byte chunk of the row piece
        const int rsub = gt >> 3;           // rows rsub + 16 i
        int stage = 0;
        uint32_t phase = 0;
        int qi = 0;
        uint32_t qph = 0;
        for (;;) {
            int tile = 0, got = 1;
            if (lane == 0) {
                if (mbar_wait_bounded_cluster(&q_full[qi], qph, s_abort, p.dev_status)) {
                    tile = q_tile[qi];
                    mbar_arrive_cluster(lead_qempty + 8u * static_cast<uint32_t>(qi));
                } else {
                    got = 0;
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (++qi == QD) {
                qi = 0;
                qph ^= 1;
            }
            if (!got || tile >= total) break;
            const Tile t = decode_tile_pair(p, tile, s_off, s_prefix, total0, 1);
            const int nrows = t.half ? 64 : 128;
            const int arow = t.row0 + nrows * static_cast<int>(rank);
            const bool seg0 = t.seg == 0;
            const int K = seg0 ? p.K0 : p.K1;
            // rows past the problem's end read its last row (their results are not stored)
            const int nlim = seg0 ? p.rows0 : p.rows1;
            const uint16_t *src[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = min(arow + rsub + 16 * i, nlim - 1);
                int sr = r;
                if (seg0) sr = min(max(__ldg(p.ga_rows0 + r), 0), p.ga_n0 - 1);
                src[i] = (seg0 ? p.gA0 : p.gA1) + static_cast<size_t>(sr) * K + 8 * j;
            }
            bool ok = true;
            for (int kb = 0; kb < t.kblocks; ++kb) {
                int e_ok = 1;
                if (lane == 0)
                    e_ok = mbar_wait_bounded(&empty[stage], phase ^ 1, s_abort, p.dev_status);
                if (!__shfl_sync(0xffffffffu, e_ok, 0)) {
                    ok = false;
                    break;
                }
                uint8_t *a_dst = smem + stage * W_STAGE_BYTES;
                const int k0 = kb * BK;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (16 * i >= nrows) break;
                    const int r = rsub + 16 * i;
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(
                                     a_dst + (r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4))),
                                 "l"(reinterpret_cast<uint64_t>(src[i] + k0))
                                 : "memory");
                }
                cp_async_mbar_arrive(&a_full[stage]);
                if (++stage == WSTAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // none of this thread's copies in flight
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM2_COLS);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// bf16 tensor [outer...][inner] viewed as K-major tiles of box_rows x 64.
bool make_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[3], gstride[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
    gstride[0] = dims[0] * 2;
    if (rank == 3) gstride[1] = dims[0] * dims[1] * 2;
    box[0] = BK;
    box[1] = static_cast<cuuint32_t>(box_rows);
    box[2] = 1;
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr),
                          gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output [rows, cols] (row stride ld elements, bf16 or fp32) as 32-row x
// 64-byte boxes with the 64-byte swizzle, for the pair kernel's TMA stores.
bool make_out_map(CUtensorMap *m, void *ptr, int rows, int cols, int64_t ld, bool f32) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int esz = f32 ? 4 : 2;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(std::max(rows, 1))};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / esz), 32};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r =
        fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, gdim,
           gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Both output maps of a launch (a missing segment reuses the other's map).
bool make_out_maps(Params &p, int cols0, int cols1) {
    const bool have0 = p.G > 0, have1 = p.rows1 > 0;
    if (have0 && !make_out_map(&p.tmO0, p.out0, p.rows0, cols0, p.ldo0, p.out0_f32 != 0))
        return false;
    if (have1 && !make_out_map(&p.tmO1, p.out1, p.rows1, cols1, p.ldo1, p.out1_f32 != 0))
        return false;
    if (!have0) p.tmO0 = p.tmO1;
    if (!have1) p.tmO1 = p.tmO0;
    return true;
}

// Which grouped-GEMM kernel runs: MOE_GEMM_KERNEL=pair or =single in the
// environment (read once) forces one; the default picks per launch.
enum GemmChoice { GEMM_AUTO, GEMM_PAIR, GEMM_SINGLE, GEMM_WIDE };
GemmChoice gemm_choice() {
    static const GemmChoice c = [] {
        const char *v = getenv("MOE_GEMM_KERNEL");
        if (v && v[0] == 'p') return GEMM_PAIR;
        if (v && v[0] == 's') return GEMM_SINGLE;
        if (v && v[0] == 'w') return GEMM_WIDE;
        return GEMM_AUTO;
    }();
    return c;
}

// The wide pair kernel takes the launches the CTA-pair kernel would (about
// 1024 rows per group or more) when the shapes give whole 512-column tiles
// (256 act columns in SwiGLU mode) in both segments: measured on GB300 with
// the clock power-capped, it runs the image-gen block's matmuls 1-1.5% and
// the skewed load's 1.7% faster than the 256 x 256 pair tiles (fewer bytes
// staged per flop, so a higher clock under the same power).  With a few
// hundred rows per group the one-CTA kernel stays faster.
bool use_wide(bool swiglu, int N, int K, const GemmSegment1 &seg1, int n, int G) {
    const GemmChoice c = gemm_choice();
    if (c == GEMM_PAIR || c == GEMM_SINGLE) return false;
    const int unit = swiglu ? 256 : 512;
    const bool fits = N % unit == 0 && K % BK == 0 &&
                      (seg1.rows == 0 || (seg1.N1 % unit == 0 && seg1.K1 % BK == 0));
    if (!fits) return false;
    if (c == GEMM_WIDE) return true;
    const int64_t avg = G > 0 ? n / G : seg1.rows;
    return avg >= 1024;
}

// 256-row pair tiles pay off when groups are large.  Each group's last
// block is padded to the tile height, so with a few hundred rows per group
// (about 512 measured: 25% padding at 256 rows, 13% at 128) and in weight
// streaming the 128-row one-CTA tiles are faster; at 2048 rows per group the
// pair kernel is.
bool use_pair(int n, int G, int seg1_rows) {
    const GemmChoice c = gemm_choice();
    if (c != GEMM_AUTO) return c == GEMM_PAIR;
    const int64_t avg = G > 0 ? n / G : seg1_rows;
    return avg >= 1024;
}

template <int MODE, int BN>
cudaError_t launch(Params &p, int max_rows0, cudaStream_t stream) {
    using C = Cfg<BN>;
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, BN>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 C::SMEM);
            if (e != cudaSuccess) return e;
            attr_done[dev] = true;
        }
    }
    // an upper bound on the tile count: sum over groups of ceil(rows/128)
    const int64_t mblocks0 = ceil_div(max_rows0, BM) + p.G;
    const int64_t tiles = mblocks0 * p.nt0 + (p.rows1 > 0 ? ceil_div(p.rows1, BM) * p.nt1 : 0);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms(), tiles)));
    grouped_gemm_kernel<MODE, BN><<<grid, THREADS, C::SMEM, stream>>>(p);
    return cudaGetLastError();
}

// Tile counters of the pair kernel.  Each launch takes the next slot of a
// ring of counters that live in the library's own device memory (no
// allocation, graph-capturable) and zeroes it on its stream right before the
// kernel.  Launches in flight at the same time (different streams) get
// different slots as long as fewer than kTileCounters of them overlap.
constexpr int kTileCounters = 256;
constexpr int kMaxDev = 64;
static __device__ unsigned int g_tile_counters[kTileCounters];

struct CounterRing {
    std::once_flag once;
    unsigned int *base = nullptr;
    cudaError_t err = cudaSuccess;
    std::atomic<unsigned int> next{0};
};
CounterRing g_rings[kMaxDev];

cudaError_t next_tile_counter(unsigned int **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    CounterRing &r = g_rings[dev];
    std::call_once(r.once, [&r] {
        void *ptr = nullptr;
        r.err = cudaGetSymbolAddress(&ptr, g_tile_counters);
        if (r.err == cudaSuccess) r.base = static_cast<unsigned int *>(ptr);
    });
    if (r.err != cudaSuccess) return r.err;
    *out = r.base + (r.next.fetch_add(1u, std::memory_order_relaxed) % kTileCounters);
    return cudaSuccess;
}

template <int MODE>
cudaError_t launch_pair(Params &p, int max_rows0, cudaStream_t stream) {
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<MODE>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Cfg2::SMEM);
            if (e != cudaSuccess) return e;
            attr_done[dev] = true;
        }
    }
    const int64_t mblocks0 = ceil_div(max_rows0, BM2) + p.G;
    const int64_t tiles = mblocks0 * p.nt0 + (p.rows1 > 0 ? ceil_div(p.rows1, BM2) * p.nt1 : 0);
    // Launch no more clusters than can be resident at once (CTA pairs need
    // two SMs of one TPC, so this can be below num_sms / 2): a persistent
    // cluster that waits for a free TPC only delays the tail.
    static int max_clusters[64] = {};
    if (dev < 64 && max_clusters[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms()), 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg2::SMEM;
        cfg.stream = stream;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<MODE>, &cfg) != cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            n = num_sms() / 2;
        }
        max_clusters[dev] = std::min(n, num_sms() / 2);
        const char *dbg = getenv("MOE_DEBUG");
        if (dbg && dbg[0] == '1')
            fprintf(stderr, "libmoe: device %d: %d CTA-pair clusters resident at once (%d SMs)\n",
                    dev, max_clusters[dev], num_sms());
    }
    const int limit = dev < 64 ? max_clusters[dev] : num_sms() / 2;
    const int clusters = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(limit, tiles)));
    cudaError_t e = next_tile_counter(&p.tile_counter);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p.tile_counter, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    grouped_gemm_pair_kernel<MODE><<<2 * clusters, THREADS, Cfg2::SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <int MODE, bool GATHER>
cudaError_t launch_wide(Params &p, int max_rows0, cudaStream_t stream) {
    constexpr int NT = GATHER ? W_THREADS_G : W_THREADS;
    static std::mutex mu;
    static bool attr_done[64] = {};
    static int max_clusters[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(grouped_gemm_wide_kernel<MODE, GATHER>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 CfgW::SMEM);
            if (e != cudaSuccess) return e;
            attr_done[dev] = true;
        }
        if (dev < 64 && max_clusters[dev] == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(num_sms()), 1, 1);
            cfg.blockDim = dim3(NT, 1, 1);
            cfg.dynamicSmemBytes = CfgW::SMEM;
            cfg.stream = stream;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_wide_kernel<MODE, GATHER>, &cfg) !=
                    cudaSuccess ||
                n <= 0) {
                cudaGetLastError();
                n = num_sms() / 2;
            }
            max_clusters[dev] = std::min(n, num_sms() / 2);
        }
    }
    const int64_t mblocks0 = ceil_div(max_rows0, BM2) + p.G;
    const int64_t tiles = mblocks0 * p.nt0 + (p.rows1 > 0 ? ceil_div(p.rows1, BM2) * p.nt1 : 0);
    const int limit = dev < 64 ? max_clusters[dev] : num_sms() / 2;
    const int clusters = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(limit, tiles)));
    cudaError_t e = next_tile_counter(&p.tile_counter);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p.tile_counter, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    grouped_gemm_wide_kernel<MODE, GATHER><<<2 * clusters, NT, CfgW::SMEM, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool tensor_maps_available() { return encode_fn() != nullptr; }

bool gemm_can_gather(int n, int G, int K, int N, const GemmSegment1 &seg1) {
    return use_wide(true, N, K, seg1, n, G) && K % 8 == 0 && (seg1.rows == 0 || seg1.K1 % 8 == 0);
}

cudaError_t launch_gemm_swiglu(const uint16_t *A, const int32_t *offsets, int G, int n, int K,
                               const uint16_t *W13, int N, uint16_t *act,
                               const GemmSegment1 &seg1, int32_t *dev_status,
                               cudaStream_t stream, const uint16_t *gather_src,
                               const int32_t *gather_rows, int gather_n) {
    if (G > MAX_GROUPS) return cudaErrorInvalidValue;
    const bool gather = gather_src != nullptr;
    if (gather && (!gather_rows || gather_n <= 0 || !gemm_can_gather(n, G, K, N, seg1)))
        return cudaErrorInvalidValue;
    Params p{};
    // the pair kernel's stages hold 128 columns of K
    const bool pair = use_pair(n, G, seg1.rows) && K % 128 == 0 &&
                      (seg1.rows == 0 || seg1.K1 % 128 == 0);
    if (G > 0) {
        const uint64_t a0[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(std::max(n, 1))};
        const uint64_t b0[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(2 * N),
                                static_cast<uint64_t>(G)};
        // gathered A: the rows are not a tensor; the B map stands in for the unused A map
        if ((!gather && !make_map(&p.tmA0, A, 2, a0, BM)) || !make_map(&p.tmB0, W13, 3, b0, 128))
            return cudaErrorInvalidValue;
        if (gather) p.tmA0 = p.tmB0;
        p.tmA1 = p.tmA0;
        p.tmB1 = p.tmB0;
    }
    if (seg1.rows > 0) {
        const uint64_t a1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.rows)};
        const uint64_t b1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(2 * seg1.N1)};
        if (!make_map(&p.tmA1, seg1.A, 2, a1, BM) || !make_map(&p.tmB1, seg1.B, 2, b1, 128))
            return cudaErrorInvalidValue;
        if (G == 0) {   // no routed groups: the unused maps just need to be valid
            p.tmA0 = p.tmA1;
            p.tmB0 = p.tmB1;
        }
    } else if (G == 0) {
        return cudaSuccess;
    }
    p.gA0 = gather_src;
    p.ga_rows0 = gather_rows;
    p.ga_n0 = gather_n;
    p.gA1 = seg1.A;
    p.offsets = offsets;
    p.G = G;
    p.rows0 = n;
    p.K0 = K;
    p.K1 = seg1.K1;
    p.nt0 = N / 128;
    p.nt1 = seg1.N1 / 128;
    p.half0 = N;
    p.half1 = seg1.N1;
    p.brows0 = 2 * N;
    p.brows1 = 2 * seg1.N1;
    p.rows1 = seg1.rows;
    p.out0 = act;
    p.ldo0 = N;
    p.out1 = seg1.out;
    p.ldo1 = seg1.N1;
    p.out0_f32 = 0;
    p.out1_f32 = 0;
    p.dev_status = dev_status;
    if (use_wide(true, N, K, seg1, n, G)) {
        // 256 act columns per tile; A as 128- and 64-row boxes, B as 256-row
        // boxes (and 64-row boxes for the gate/up quarters of half tiles)
        p.nt0 = N / 256;
        p.nt1 = seg1.N1 / 256;
        if (!make_out_maps(p, N, seg1.N1)) return cudaErrorInvalidValue;
        if (G > 0) {
            const uint64_t a0[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(std::max(n, 1))};
            const uint64_t b0[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(2 * N),
                                    static_cast<uint64_t>(G)};
            if ((!gather && !make_map(&p.tmA0h, A, 2, a0, 64)) ||
                !make_map(&p.tmB0h, W13, 3, b0, 64) || !make_map(&p.tmB0w, W13, 3, b0, 256))
                return cudaErrorInvalidValue;
            if (gather) p.tmA0h = p.tmB0h;
        }
        if (seg1.rows > 0) {
            const uint64_t a1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.rows)};
            const uint64_t b1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(2 * seg1.N1)};
            if (!make_map(&p.tmA1h, seg1.A, 2, a1, 64) || !make_map(&p.tmB1h, seg1.B, 2, b1, 64) ||
                !make_map(&p.tmB1w, seg1.B, 2, b1, 256))
                return cudaErrorInvalidValue;
        }
        if (G == 0) {
            p.tmA0h = p.tmA1h;
            p.tmB0h = p.tmB1h;
            p.tmB0w = p.tmB1w;
        }
        if (seg1.rows == 0) {
            p.tmA1h = p.tmA0h;
            p.tmB1h = p.tmB0h;
            p.tmB1w = p.tmB0w;
        }
        return gather ? launch_wide<MODE_SWIGLU, true>(p, n, stream)
                      : launch_wide<MODE_SWIGLU, false>(p, n, stream);
    }
    if (pair) {
        if (!make_out_maps(p, N, seg1.N1)) return cudaErrorInvalidValue;
        // 64-row boxes for half tiles: A, and B as 64 gate + 64 up rows
        if (G > 0) {
            const uint64_t a0[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(std::max(n, 1))};
            const uint64_t b0[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(2 * N),
                                    static_cast<uint64_t>(G)};
            if (!make_map(&p.tmA0h, A, 2, a0, 64) || !make_map(&p.tmB0h, W13, 3, b0, 64))
                return cudaErrorInvalidValue;
        }
        if (seg1.rows > 0) {
            const uint64_t a1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.rows)};
            const uint64_t b1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(2 * seg1.N1)};
            if (!make_map(&p.tmA1h, seg1.A, 2, a1, 64) || !make_map(&p.tmB1h, seg1.B, 2, b1, 64))
                return cudaErrorInvalidValue;
        }
        if (G == 0) {
            p.tmA0h = p.tmA1h;
            p.tmB0h = p.tmB1h;
        }
        if (seg1.rows == 0) {
            p.tmA1h = p.tmA0h;
            p.tmB1h = p.tmB0h;
        }
        return launch_pair<MODE_SWIGLU>(p, n, stream);
    }
    return launch<MODE_SWIGLU, 256>(p, n, stream);
}

cudaError_t launch_gemm_store(const uint16_t *A, const int32_t *offsets, int G, int n, int K,
                              const uint16_t *W, int N, void *y, const GemmSegment1 &seg1,
                              int32_t *dev_status, cudaStream_t stream, bool y_f32) {
    if (G > MAX_GROUPS) return cudaErrorInvalidValue;
    const int BN = (N % 256 == 0 && (seg1.rows == 0 || seg1.N1 % 256 == 0)) ? 256 : 128;
    const bool pair = BN == 256 && use_pair(n, G, seg1.rows) && K % 128 == 0 &&
                      (seg1.rows == 0 || seg1.K1 % 128 == 0);
    const int box_b = pair ? 128 : BN;   // a pair CTA stages half of the 256 B rows
    Params p{};
    if (G > 0) {
        const uint64_t a0[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(std::max(n, 1))};
        const uint64_t b0[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                                static_cast<uint64_t>(G)};
        if (!make_map(&p.tmA0, A, 2, a0, BM) || !make_map(&p.tmB0, W, 3, b0, box_b))
            return cudaErrorInvalidValue;
        p.tmA1 = p.tmA0;
        p.tmB1 = p.tmB0;
    }
    if (seg1.rows > 0) {
        const uint64_t a1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.rows)};
        const uint64_t b1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.N1)};
        if (!make_map(&p.tmA1, seg1.A, 2, a1, BM) || !make_map(&p.tmB1, seg1.B, 2, b1, box_b))
            return cudaErrorInvalidValue;
        if (G == 0) {
            p.tmA0 = p.tmA1;
            p.tmB0 = p.tmB1;
        }
    } else if (G == 0) {
        return cudaSuccess;
    }
    p.offsets = offsets;
    p.G = G;
    p.rows0 = n;
    p.K0 = K;
    p.K1 = seg1.K1;
    p.nt0 = N / BN;
    p.nt1 = seg1.N1 / BN;
    p.half0 = 0;
    p.half1 = 0;
    p.brows0 = N;
    p.brows1 = seg1.N1;
    p.rows1 = seg1.rows;
    p.out0 = y;
    p.ldo0 = N;
    p.out1 = seg1.out;
    p.ldo1 = seg1.N1;
    p.out0_f32 = y_f32 ? 1 : 0;
    p.out1_f32 = seg1.out_f32 ? 1 : 0;
    p.dev_status = dev_status;
    if (use_wide(false, N, K, seg1, n, G)) {
        // 512 output columns per tile; A as 128- and 64-row boxes, B as
        // 256-row boxes
        p.nt0 = N / 512;
        p.nt1 = seg1.N1 / 512;
        if (!make_out_maps(p, N, seg1.N1)) return cudaErrorInvalidValue;
        if (G > 0) {
            const uint64_t a0[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(std::max(n, 1))};
            const uint64_t b0[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                                    static_cast<uint64_t>(G)};
            if (!make_map(&p.tmA0h, A, 2, a0, 64) || !make_map(&p.tmB0w, W, 3, b0, 256))
                return cudaErrorInvalidValue;
        }
        if (seg1.rows > 0) {
            const uint64_t a1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.rows)};
            const uint64_t b1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.N1)};
            if (!make_map(&p.tmA1h, seg1.A, 2, a1, 64) || !make_map(&p.tmB1w, seg1.B, 2, b1, 256))
                return cudaErrorInvalidValue;
        }
        if (G == 0) {
            p.tmA0h = p.tmA1h;
            p.tmB0w = p.tmB1w;
        }
        if (seg1.rows == 0) {
            p.tmA1h = p.tmA0h;
            p.tmB1w = p.tmB0w;
        }
        p.tmB0h = p.tmB0w;
        p.tmB1h = p.tmB1w;
        return launch_wide<MODE_STORE, false>(p, n, stream);
    }
    if (pair) {
        if (!make_out_maps(p, N, seg1.N1)) return cudaErrorInvalidValue;
        // 64-row A boxes for half tiles (B keeps its 128-row boxes)
        if (G > 0) {
            const uint64_t a0[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(std::max(n, 1))};
            if (!make_map(&p.tmA0h, A, 2, a0, 64)) return cudaErrorInvalidValue;
        }
        if (seg1.rows > 0) {
            const uint64_t a1[2] = {static_cast<uint64_t>(seg1.K1), static_cast<uint64_t>(seg1.rows)};
            if (!make_map(&p.tmA1h, seg1.A, 2, a1, 64)) return cudaErrorInvalidValue;
        }
        if (G == 0) p.tmA0h = p.tmA1h;
        if (seg1.rows == 0) p.tmA1h = p.tmA0h;
        p.tmB0h = p.tmB0;
        p.tmB1h = p.tmB1;
        return launch_pair<MODE_STORE>(p, n, stream);
    }
    if (BN == 256) return launch<MODE_STORE, 256>(p, n, stream);
    return launch<MODE_STORE, 128>(p, n, stream);
}

}  // namespace moe
