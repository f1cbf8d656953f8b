// Block-scaled FP4 GEMM on a CTA pair: the same product as gemm.cu,
//
//   Y[m, n] = bf16( g_a * g_b * sum_k e2m1(A[m,k]) e4m3(SA[m,k/16])
//                                     e2m1(B[n,k]) e4m3(SB[n,k/16]) )
//
// (the "nvfp4-difusion" page's quantized matmul, section 2), computed with
// the two-SM form of the tensor-core instruction (tcgen05 .cta_group::2).
//
// Why a pair: one 128 x 256 x 64 FP4 MMA takes 128 cycles, so a single SM
// with a 128 x 256 tile must receive 48 KiB of A/B (+6 KiB of scales) every
// 512 cycles, more than TMA delivers into one SM's shared memory when all
// SMs stream at once. In a pair each CTA holds 128 rows of A and 128 rows
// of B of a 256 x 256 tile and the instruction reads the partner's half of
// B directly, so each SM receives 32 KiB of A/B per 512 MMA cycles.
//
// Persistent kernel, clusters of 2 CTAs (one per SM), 256 x 256 output
// tiles per pair, K in stages of 256 (4 MMAs of K = 64). Warp roles, in
// both CTAs unless noted:
//   warp 0    TMA producer of this CTA's 128 A rows and 128 B rows of stage g
//             into a STAGES-deep ring;
//   warp 2    allocates / frees TMEM (jointly with the partner CTA), and is
//             the TMA producer of the stage's scales: this CTA's A scales
//             and all 256 B-row scales of the tile (one 3-D box). Every load
//             of both CTAs is counted on the full barrier of rank 0;
//   warp 1    (rank 0) MMA issuer: per stage and K = 64 step, 3 scale
//             copies shared -> TMEM and 1 MMA, each one instruction for both
//             CTAs; the release of the stage and of the finished
//             accumulator is multicast to both CTAs' barriers;
//   warps 3-10 epilogue over this CTA's 128 accumulator rows: tcgen05.ld,
//             release to rank 0's accumulator barrier (16 arrivals: 8 warps
//             x 2 CTAs), scale by g_a g_b, round to bfloat16, store.
// The copies stay in the MMA thread: a separate copy warp synchronised by
// tcgen05.commit let the partner SM's MMA read a scale replica before its
// copy had landed (wrong products in one TMEM lane quarter); from one
// thread, copy and MMA reach both SMs in issue order. Two producer warps
// halve the TMA issue work per warp.
// Every mbarrier wait is bounded in time; a wait that runs out records a
// timeout in the device error word and the roles of both CTAs leave.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"
#include "tensor_map.h"

namespace nvfp4 {

namespace {

constexpr int PM = 256;                    // tile rows per pair
constexpr int BM = 128;                    // ... per CTA
constexpr int BN = 256;                    // tile columns
constexpr int BNH = 128;                   // B rows loaded by each CTA
constexpr int BK = 256;                    // FP4 elements per stage
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * BK / 2;       // 16 KiB
constexpr int B_BYTES = BNH * BK / 2;      // 16 KiB
constexpr int SFA_BYTES = BM * BK / 16;    // 2 KiB: 4 tiles of 512 B
constexpr int SFB_BYTES = BN * BK / 16;    // 4 KiB: 2 row groups x 4 tiles
constexpr int SF_TILE = 512;
constexpr int SF_ROW = 256;                // scale arrays as rows of 256 bytes
constexpr int CTA_STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr uint32_t STAGE_TX = 2 * CTA_STAGE_BYTES;  // both CTAs, counted at rank 0
// a stage of a column-half unit (256 x 128): each CTA loads 64 B rows
constexpr uint32_t STAGE_TX_HALF = 2 * (CTA_STAGE_BYTES - B_BYTES / 2);
// LoRA stage (after a tile's FP4 stages): L' (128 rows x 64 bfloat16) in the
// A slot, the up projection (128 rows x 64 bfloat16) in the B slot, no scales
constexpr uint32_t LORA_TX = 2 * (A_BYTES + B_BYTES);
constexpr int MMAS_PER_STAGE = BK / 64;    // 4
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;            // 256 FP32 columns
constexpr uint32_t SF_COL = 256;           // per stage: 16 (SFA) + 32 (SFB)
constexpr uint32_t SF_COLS_PER_STAGE = 48;
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 3;
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);  // 352
constexpr int GROUP_M = 8;                 // raster: 8 pair rows (2048 rows) per sweep
constexpr uint16_t kPairMask = 0x3;
constexpr unsigned kAll = 0xFFFFFFFFu;

constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
constexpr int SMEM_SFA = SMEM_B + STAGES * B_BYTES;
constexpr int SMEM_SFB = SMEM_SFA + STAGES * SFA_BYTES;
constexpr int EPI_CHUNK = 64;              // output columns per TMA store (128 B rows)
constexpr int EPI_BYTES = 32 * EPI_CHUNK * 2;  // one warp's 32 rows x 64 columns of bfloat16
constexpr int SMEM_EPI = SMEM_SFB + STAGES * SFB_BYTES;  // 1024-aligned staging, one per warp
constexpr int SMEM_BAR = SMEM_EPI + kEpiWarps * EPI_BYTES;
constexpr int SMEM_RTAB = SMEM_BAR + 256;  // re-quantization: 1 / (e4m3(S) g_y) for the 128 S
constexpr int SMEM_USED = SMEM_RTAB + 128 * 4;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // room to align the base to 1024

static_assert(SF_COL + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
static_assert(SMEM_EPI % 1024 == 0 && EPI_BYTES % 1024 == 0, "128-byte swizzle atoms");

struct Params {
    const float *g_a;
    const float *g_b;
    uint16_t *Y;
    int64_t ldy;
    int M, N, K;
    int num_m_tiles;     // 256-row tiles
    int num_n_tiles;     // 256-column tiles
    int num_tiles;
    int y_vec;           // rows of Y start 16-byte aligned: 16-byte stores
    int y_tma;           // Y written by TMA stores (rows 16-byte aligned, map valid)
    int store_y;         // 0: Y is not written (re-quantized output only)
    const uint16_t *bias;  // optional bfloat16 bias, N values
    // optional output re-quantization (N % 256 == 0): the bfloat16 Y values
    // quantized with g_y into codes (M x N/2) and tile-layout scales (rows
    // padded to 128), as nvfp4_quantize would
    const float *g_y;
    uint8_t *Yq;
    uint8_t *Ys;
    WeightGroups groups;  // grouped projection: g_b holds one scale per group
    int lora_r;           // > 0: one LoRA stage of lora_r / 16 bfloat16 K-steps per tile
    // Work units: [0, num_full) are whole 256 x 256 tiles; the remaining
    // tiles (the partial last wave) run as two 256 x 128 column halves each
    // (N = 128 MMAs on otherwise idle pairs; the same K order, so the same
    // bits per element).
    int num_full;
    int num_units;
    uint32_t *y_amax;    // kMode 2: max |y| of the stored output (rows < M), atomically
    int inject;          // 1: the producers issue nothing (bounded-wait test)
    uint64_t timeout_ns;
    unsigned int *err;   // device error word
};

struct Shared {
    uint64_t full[STAGES];   // (rank 0) both CTAs' loads of the stage landed
    uint64_t empty[STAGES];  // MMAs of the stage done: its slot may be refilled
    uint64_t acc_full;       // accumulator complete (both CTAs)
    uint64_t acc_empty;      // (rank 0) both CTAs drained the accumulator
    uint64_t drain_mma;      // teardown after an abort: MMAs issued have completed
    uint32_t tmem_base;
    volatile uint32_t abort_flag;
};
static_assert(sizeof(Shared) <= 256, "barrier area");

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int &mt, int &nt) {
    const int per_group = GROUP_M * num_n;
    const int group = t / per_group;
    const int first_m = group * GROUP_M;
    const int gsz = min(num_m - first_m, GROUP_M);
    const int local = t - group * per_group;
    mt = first_m + local % gsz;
    nt = local / gsz;
}

// Work unit u: a whole tile (half -1) or one column half (0 / 1) of a tile.
struct Unit {
    int tile, half;
};
__device__ __forceinline__ Unit unit_of(int u, const Params &p) {
    if (u < p.num_full) return {u, -1};
    const int v = u - p.num_full;
    return {p.num_full + (v >> 1), v & 1};
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Bounded wait by lane 0 of a converged warp, also giving up once another
// role of this CTA has aborted; the outcome is broadcast to the warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const Params &p,
                                          Shared &sh) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        const uint32_t a = smem_addr(bar);
        if (!mbar_try_wait(a, parity)) {
            const uint64_t t0 = global_timer_ns();
            while (true) {
                if (mbar_try_wait(a, parity)) break;
                if (sh.abort_flag) {
                    ok = 0;
                    break;
                }
                if (global_timer_ns() - t0 > p.timeout_ns) {
                    record_timeout(p.err);
                    sh.abort_flag = 1;
                    ok = 0;
                    break;
                }
            }
        }
    }
    return __shfl_sync(kAll, ok, 0) != 0;
}

// kMode 0: the plain epilogue; 1: the bias / re-quantization / grouped /
// LoRA epilogue; 2: that, plus the largest |y| of the output folded into
// p.y_amax. Separate instantiations, so the plainer kernels' registers are
// not spent on what they do not do.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSA,
                     const __grid_constant__ CUtensorMap tmSB,
                     const __grid_constant__ CUtensorMap tmY,
                     const __grid_constant__ CUtensorMap tmYq,
                     const __grid_constant__ CUtensorMap tmL,
                     const __grid_constant__ CUtensorMap tmLB,
                     const __grid_constant__ CUtensorMap tmB64, const Params p) {
    constexpr bool kEpi = kMode >= 1;
    constexpr bool kAmax = kMode == 2;
    // tmSA: A scales as rows of 256 B (8 rows per stage); tmSB: B scales as
    // {256 B, rows of a 128-row group, group} (8 rows x 2 groups per stage)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Shared &sh = *reinterpret_cast<Shared *>(smem + SMEM_BAR);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int my_units =
        pair < p.num_units ? (p.num_units - pair + num_pairs - 1) / num_pairs : 0;
    const int num_k = p.K / BK;
    const int kb4 = p.K / 64;  // 512-byte scale tiles per 128-row group

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.acc_full, 1);
        mbar_init(&sh.acc_empty, 2 * kEpiWarps);
        mbar_init(&sh.drain_mma, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (p.num_units > p.num_full) tma_prefetch_desc(&tmB64);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
        if (p.y_tma) tma_prefetch_desc(&tmY);
        if (kEpi && p.Yq != nullptr) tma_prefetch_desc(&tmYq);
        if (kEpi && p.lora_r > 0) {
            tma_prefetch_desc(&tmL);
            tma_prefetch_desc(&tmLB);
        }
    }
    if (warp == 2) {
        tmem_alloc_pair(&sh.tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers and TMEM exist before any remote use
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0 || warp == 2) {
        // --------------------------------------- TMA producers (A/B; scales)
        const bool scales = warp == 2;
        const uint64_t pol = policy_evict_last();
        const uint32_t full0 = mapa_shared(smem_addr(&sh.full[0]), 0);
        int g = 0;
        bool ok = !p.inject;
        for (int t = 0; ok && t < my_units; ++t) {
            const Unit un = unit_of(pair + t * num_pairs, p);
            const bool hu = un.half >= 0;
            int mt, nt;
            tile_coords(un.tile, p.num_m_tiles, p.num_n_tiles, mt, nt);
            const int arow = mt * PM + static_cast<int>(rank) * BM;
            // B rows of this CTA: 128 of the tile's 256, or 64 of a half's 128
            const int brow = hu ? nt * BN + un.half * BNH + static_cast<int>(rank) * (BNH / 2)
                                : nt * BN + static_cast<int>(rank) * BNH;
            const int sfb_group = nt * 2 + (hu ? un.half : 0);
            // scale rows of 256 B: group grp, stage kt starts at row
            // (grp * kb4 + 4 kt) * 2; groups past the array read as 0
            const int sfa_row = (mt * 2 + static_cast<int>(rank)) * kb4 * 2;
            for (int kt = 0; kt < num_k; ++kt, ++g) {
                const int s = g % STAGES;
                if (!warp_wait(&sh.empty[s], ((g / STAGES) & 1) ^ 1, p, sh)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t bar = full0 + static_cast<uint32_t>(s) * 8u;
                    if (!scales) {
                        if (leader)
                            mbar_arrive_expect_tx(&sh.full[s], hu ? STAGE_TX_HALF : STAGE_TX);
                        tma_load_2d_pair(smem + SMEM_A + s * A_BYTES, &tmA, bar, kt * (BK / 2),
                                         arow, pol);
                        tma_load_2d_pair(smem + SMEM_B + s * B_BYTES, hu ? &tmB64 : &tmB, bar,
                                         kt * (BK / 2), brow, pol);
                    } else {
                        tma_load_2d_pair(smem + SMEM_SFA + s * SFA_BYTES, &tmSA, bar, 0,
                                         sfa_row + kt * 8, pol);
                        tma_load_3d_pair(smem + SMEM_SFB + s * SFB_BYTES, &tmSB, bar, 0, kt * 8,
                                         sfb_group, pol);
                    }
                }
                __syncwarp();
            }
            if (kEpi && ok && p.lora_r > 0) {
                // the tile's LoRA stage: A/B producer only (no scales)
                const int s = g % STAGES;
                if (!scales) {
                    if (!warp_wait(&sh.empty[s], ((g / STAGES) & 1) ^ 1, p, sh)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const uint32_t bar = full0 + static_cast<uint32_t>(s) * 8u;
                        if (leader) mbar_arrive_expect_tx(&sh.full[s], LORA_TX);
                        tma_load_2d_pair(smem + SMEM_A + s * A_BYTES, &tmL, bar, 0, arow, pol);
                        tma_load_2d_pair(smem + SMEM_B + s * B_BYTES, &tmLB, bar, 0, brow, pol);
                    }
                    __syncwarp();
                }
                ++g;
            }
        }
        if (ok) {
            // the last releases multicast to this CTA land before it exits
            for (int s = 0; s < STAGES && s < g; ++s) {
                const int fills = (g - s + STAGES - 1) / STAGES;
                if (!warp_wait(&sh.empty[s], (fills - 1) & 1, p, sh)) break;
            }
        }
        if (!ok && !p.inject && leader && lane == 0 && !scales) {
            // let loads already issued land before the CTA exits
            for (int s = 0; s < STAGES && s < g; ++s) {
                const int fills = (g - s + STAGES - 1) / STAGES;
                mbar_wait(&sh.full[s], (fills - 1) & 1, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1 && leader) {
        // ------------------------------------------- MMA issuer (rank 0)
        constexpr uint32_t idesc_full = idesc_mxf4nvf4(PM, BN);
        constexpr uint32_t idesc_half = idesc_mxf4nvf4(PM, BN / 2);
        int g = 0, it = 0;
        bool ok = true;
        for (int t = 0; ok && t < my_units; ++t, ++it) {
            const uint32_t idesc = unit_of(pair + t * num_pairs, p).half >= 0 ? idesc_half
                                                                              : idesc_full;
            if (!warp_wait(&sh.acc_empty, (it & 1) ^ 1, p, sh)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kt = 0; kt < num_k; ++kt, ++g) {
                const int s = g % STAGES;
                if (!warp_wait(&sh.full[s], (g / STAGES) & 1, p, sh)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // per K = 64 step: the step's scales shared -> TMEM for both
                // CTAs, then the MMA that reads them, in issue order
                const uint32_t sf_a = tmem + SF_COL + s * SF_COLS_PER_STAGE;
                const uint32_t sf_b = sf_a + 16;
                const uint32_t sfa_smem = smem_addr(smem + SMEM_SFA + s * SFA_BYTES);
                const uint32_t sfb_smem = smem_addr(smem + SMEM_SFB + s * SFB_BYTES);
                const uint32_t a_smem = smem_addr(smem + SMEM_A + s * A_BYTES);
                const uint32_t b_smem = smem_addr(smem + SMEM_B + s * B_BYTES);
#pragma unroll
                for (int j = 0; j < MMAS_PER_STAGE; ++j)
                    sf_copy3_mma_pair_elect(tmem + ACC_COL, sdesc_sw128(a_smem + j * 32),
                                            sdesc_sw128(b_smem + j * 32), idesc, sf_a + j * 4,
                                            sf_b + j * 8, (kt | j) != 0,
                                            sdesc_sf(sfa_smem + j * SF_TILE),
                                            sdesc_sf(sfb_smem + j * SF_TILE),
                                            sdesc_sf(sfb_smem + SFB_BYTES / 2 + j * SF_TILE));
                tc_commit_pair_mc_elect(&sh.empty[s], kPairMask);
            }
            if (kEpi && ok && p.lora_r > 0) {
                // LoRA up projection into the same accumulator: L' (this
                // pair's 256 rows x r) times the up-projection rows (256 x r),
                // r / 16 bfloat16 K-steps of 32 bytes in the swizzled rows
                constexpr uint32_t idesc_l = idesc_bf16(PM, BN);
                const int s = g % STAGES;
                if (!warp_wait(&sh.full[s], (g / STAGES) & 1, p, sh)) {
                    ok = false;
                } else {
                    tc_fence_after();
                    const uint32_t a_smem = smem_addr(smem + SMEM_A + s * A_BYTES);
                    const uint32_t b_smem = smem_addr(smem + SMEM_B + s * B_BYTES);
                    for (int j = 0; j < p.lora_r / 16; ++j)
                        mma_bf16_pair_elect(tmem + ACC_COL, sdesc_sw128(a_smem + j * 32),
                                            sdesc_sw128(b_smem + j * 32), idesc_l, 1u);
                    tc_commit_pair_mc_elect(&sh.empty[s], kPairMask);
                    ++g;
                }
            }
            if (ok) tc_commit_pair_mc_elect(&sh.acc_full, kPairMask);
        }
        if (!ok) {
            // MMAs already issued must complete before TMEM is released
            tc_commit_pair_mc_elect(&sh.drain_mma, 0x1);
            if (lane == 0) mbar_wait(&sh.drain_mma, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp >= kFirstEpiWarp) {
        // -------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int half = (warp - kFirstEpiWarp) >> 2;  // which 128 columns
        const float g_a = *p.g_a;
        const float alpha0 = __fmul_rn(g_a, *p.g_b);
        const uint32_t acc_empty0 = mapa_shared(smem_addr(&sh.acc_empty), 0);
        // re-quantization: the block multiplier for each of the 128 scale
        // bytes, filled once by the epilogue warps (the standalone
        // quantizer's table, the same IEEE operations)
        float *rtab = reinterpret_cast<float *>(smem + SMEM_RTAB);
        const float gy = (kEpi && p.Yq != nullptr) ? *p.g_y : 1.0f;
        if (kEpi && p.Yq != nullptr) {
            for (int i = threadIdx.x - 32 * kFirstEpiWarp; i < 128; i += 32 * kEpiWarps)
                rtab[i] = scale_recip(static_cast<uint32_t>(i), gy);
            asm volatile("bar.sync 2, %0;" ::"n"(32 * kEpiWarps) : "memory");
        }
        int it = 0;
        for (int t = 0; t < my_units; ++t, ++it) {
            const Unit un = unit_of(pair + t * num_pairs, p);
            if (!warp_wait(&sh.acc_full, it & 1, p, sh)) break;
            tc_fence_after();
            if (un.half >= 0 && half == 1) {
                // a column-half unit fills accumulator columns 0..127 only
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty0);
                continue;
            }
            int mt, nt;
            tile_coords(un.tile, p.num_m_tiles, p.num_n_tiles, mt, nt);
            const uint32_t t_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + ACC_COL +
                                    static_cast<uint32_t>(half * 128);
            // all four 32-column loads in flight, one wait, release the
            // accumulator to rank 0, then scale and round
            uint32_t r[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(t_base + c * 32, r[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty0);
            const int row0 = mt * PM + static_cast<int>(rank) * BM + quarter * 32;
            const int row = row0 + lane;
            const int n0 = nt * BN + (un.half >= 0 ? un.half : half) * 128;
            // grouped projection: the tile's weight group sets the scale
            const float alpha =
                kEpi ? __fmul_rn(g_a, p.g_b[weight_group_of(p.groups, n0)]) : alpha0;
            uint32_t packed[64];
            if (!kEpi || p.bias == nullptr) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        packed[c * 16 + i] = pack_bf16x2(__uint_as_float(r[c][2 * i]) * alpha,
                                                         __uint_as_float(r[c][2 * i + 1]) * alpha);
            } else {
                // y = acc * g_a g_b + bias[n] in fp32, then one rounding
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const int col = n0 + c * 32 + q8 * 8;
                        uint4 bv = make_uint4(0, 0, 0, 0);
                        if (col + 8 <= p.N) bv = __ldg(reinterpret_cast<const uint4 *>(p.bias + col));
                        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int e = q8 * 8 + 2 * i;  // column within the 32-column chunk
                            packed[c * 16 + q8 * 4 + i] = pack_bf16x2(
                                __fadd_rn(__fmul_rn(__uint_as_float(r[c][e]), alpha), bf16_lo(bw[i])),
                                __fadd_rn(__fmul_rn(__uint_as_float(r[c][e + 1]), alpha),
                                          bf16_hi(bw[i])));
                        }
                    }
                }
            }
            if (kEpi && !p.store_y) {
                // re-quantized output only
            } else if (p.y_tma) {
                // 64-column chunks through this warp's staging tile (128-byte
                // swizzle: 16-byte piece k of row r sits at piece k ^ (r % 8)),
                // written out by one TMA store each; rows >= M and columns
                // >= N are clipped by the tensor map
                uint8_t *stage = smem + SMEM_EPI + (warp - kFirstEpiWarp) * EPI_BYTES;
#pragma unroll
                for (int c = 0; c < 128 / EPI_CHUNK; ++c) {
                    if (lane == 0) bulk_wait_read_all();  // previous store has read the tile
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (NVFP4_CHECK(lane * 128 + ((k ^ (lane & 7)) * 16) + 16 <= EPI_BYTES))
                            *reinterpret_cast<uint4 *>(stage + lane * 128 +
                                                       ((k ^ (lane & 7)) * 16)) =
                                make_uint4(packed[c * 32 + 4 * k], packed[c * 32 + 4 * k + 1],
                                           packed[c * 32 + 4 * k + 2], packed[c * 32 + 4 * k + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmY, stage, n0 + c * EPI_CHUNK, row0);
                        bulk_commit_group();
                    }
                }
            } else if (row < p.M) {
                uint16_t *yrow = p.Y + static_cast<int64_t>(row) * p.ldy;
                if (p.y_vec && n0 + 128 <= p.N && NVFP4_CHECK(n0 >= 0)) {
                    uint4 *dst = reinterpret_cast<uint4 *>(yrow + n0);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                            packed[4 * i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int n = n0 + 2 * i;
                        if (n < p.N) yrow[n] = static_cast<uint16_t>(packed[i] & 0xFFFFu);
                        if (n + 1 < p.N) yrow[n + 1] = static_cast<uint16_t>(packed[i] >> 16);
                    }
                }
            }
            if (kAmax && p.y_amax != nullptr) {
                // the largest |y| of this thread's row (bfloat16 magnitude
                // bits, which order like the values), one atomic per warp;
                // rows >= M hold the bias only and are not part of Y
                uint32_t m2 = 0;
                if (row < p.M) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) m2 = max_u16x2(m2, packed[i] & 0x7FFF7FFFu);
                }
                uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
                m = __reduce_max_sync(kAll, m);
                if (lane == 0 && m != 0u) atomicMax(p.y_amax, m);
            }
            if (kEpi && p.Yq != nullptr) {
                // re-quantize this thread's 128 bfloat16 values (8 blocks of
                // 16) for the next layer, after the Y stores are in flight.
                // Codes (64 bytes of the row) go through the warp's staging
                // tile (64-byte swizzle: 16-byte piece j of row r at
                // j ^ ((r / 2) % 4)) and one TMA store, which clips rows >= M;
                // scales go straight to the tile layout (4 consecutive blocks
                // = one aligned 32-bit word), 0 on padding rows M .. M
                // rounded to 128
                uint32_t code[16];
                uint32_t sw[2] = {0u, 0u};
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const uint32_t S = quantize16_tab(
                        make_uint4(packed[8 * b], packed[8 * b + 1], packed[8 * b + 2],
                                   packed[8 * b + 3]),
                        make_uint4(packed[8 * b + 4], packed[8 * b + 5], packed[8 * b + 6],
                                   packed[8 * b + 7]),
                        gy, rtab, code[2 * b], code[2 * b + 1]);
                    sw[b >> 2] |= S << (8 * (b & 3));
                }
                uint8_t *stage = smem + SMEM_EPI + (warp - kFirstEpiWarp) * EPI_BYTES;
                if (lane == 0) bulk_wait_read_all();  // the Y stores have read the tile
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (NVFP4_CHECK(lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16) + 16 <= EPI_BYTES))
                        *reinterpret_cast<uint4 *>(stage + lane * 64 +
                                                   ((j ^ ((lane >> 1) & 3)) * 16)) =
                            make_uint4(code[4 * j], code[4 * j + 1], code[4 * j + 2],
                                       code[4 * j + 3]);
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmYq, stage, n0 / 2, row0);
                    bulk_commit_group();
                }
                const int64_t rows_pad = (static_cast<int64_t>(p.M) + 127) / 128 * 128;
                if (row < rows_pad) {
                    const int kb4y = p.N / 64;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int kb = n0 / 16 + 4 * h2;  // multiple of 4
                        const int64_t off =
                            ((static_cast<int64_t>(row >> 7) * kb4y + (kb >> 2)) << 9) +
                            ((row & 31) << 4) + (((row & 127) >> 5) << 2);
                        if (NVFP4_CHECK(off + 4 <= rows_pad * (p.N / 16)))
                            *reinterpret_cast<uint32_t *>(p.Ys + off) = row < p.M ? sw[h2] : 0u;
                    }
                }
            }
        }
        if ((p.y_tma || (kEpi && p.Yq != nullptr)) && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the other may address it
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

}  // namespace

int gemm_kernel_choice() { return debug_state().gemm_kernel; }

cudaError_t launch_gemm_plain(const GemmArgs &a, cudaStream_t st) {
    return gemm_kernel_choice() == kGemmSingle ? launch_gemm(a, st) : launch_gemm_pair(a, st);
}

cudaError_t launch_gemm_pair(const GemmArgs &a, cudaStream_t st) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    static DeviceOnce once;
    static int max_clusters_of[kMaxDevices + 1] = {};
    const cudaError_t e_setup = once.run([](int slot) {
        cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<0>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_pair_kernel<1>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_pair_kernel<2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        int max_clusters = launch_cfg().num_sms / 2;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * max_clusters, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = SMEM_ALLOC;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<0>, &cfg) == cudaSuccess && n > 0 &&
            n < max_clusters)
            max_clusters = n;
        (void)cudaGetLastError();  // a failed query leaves the default
        max_clusters_of[slot] = max_clusters;
        return cudaSuccess;
    });
    if (e_setup != cudaSuccess) return e_setup;
    const int max_clusters = max_clusters_of[device_slot()];
    const int64_t kb4 = a.K / 64;
    const int64_t sf_rows_a = (a.M + 127) / 128 * kb4 * 2;  // 256-byte rows
    const int64_t groups_b = (a.N + 127) / 128;
    CUtensorMap tmA, tmB, tmSA, tmSB, tmB64;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Aq, a.K / 2, a.M, a.K / 2, 128u, BM,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Bq, a.K / 2, a.N, a.K / 2, 128u, BNH,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tmB64, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Bq, a.K / 2, a.N, a.K / 2, 128u,
                     BNH / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tmSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.As, SF_ROW, sf_rows_a, SF_ROW,
                     SF_ROW, SFA_BYTES / SF_ROW, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_3d(&tmSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Bs, SF_ROW, kb4 * 2, groups_b, SF_ROW,
                     kb4 * SF_TILE, SF_ROW, (SFB_BYTES / 2) / SF_ROW, 2))
        return cudaErrorInvalidValue;
    CUtensorMap tmY;
    const bool store_y = a.Y != nullptr;
    const bool y_vec =
        store_y && (a.ldy % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.Y) & 15) == 0);
    const bool y_tma = y_vec && make_map_2d(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.Y, a.N, a.M,
                                            a.ldy * 2, EPI_CHUNK, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!y_tma) memset(&tmY, 0, sizeof(tmY));
    // LoRA operands: L' (M x r) and the up projection (N x r), bfloat16,
    // 128-row x 64-element boxes (columns past r read as 0)
    CUtensorMap tmL, tmLB;
    memset(&tmL, 0, sizeof(tmL));
    memset(&tmLB, 0, sizeof(tmLB));
    if (a.lora_Lp != nullptr &&
        (!make_map_2d(&tmL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.lora_Lp, a.lora_r, a.M,
                      a.lora_r * 2, 64u, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map_2d(&tmLB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.lora_B, a.lora_r, a.N,
                      a.lora_r * 2, 64u, BNH, CU_TENSOR_MAP_SWIZZLE_128B)))
        return cudaErrorInvalidValue;
    // re-quantized codes: rows of N/2 bytes, 32-row x 64-byte boxes
    CUtensorMap tmYq;
    memset(&tmYq, 0, sizeof(tmYq));
    if (a.Yq != nullptr &&
        !make_map_2d(&tmYq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Yq, a.N / 2, a.M, a.N / 2, 64u, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    Params p;
    p.g_a = a.g_a;
    p.g_b = a.g_b;
    p.Y = a.Y;
    p.ldy = a.ldy;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.K = static_cast<int>(a.K);
    p.num_m_tiles = static_cast<int>((a.M + PM - 1) / PM);
    p.num_n_tiles = static_cast<int>((a.N + BN - 1) / BN);
    p.num_tiles = p.num_m_tiles * p.num_n_tiles;
    p.y_vec = y_vec;
    p.y_tma = y_tma;
    p.store_y = store_y ? 1 : 0;
    p.bias = a.bias;
    p.g_y = a.g_y;
    p.Yq = a.Yq;
    p.Ys = a.Ys;
    p.groups = a.groups;
    // the partial last wave's tiles as column halves, when they then fit in
    // one wave (plain epilogue only)
    const bool epi = !store_y || a.bias != nullptr || a.Yq != nullptr || a.groups.count > 1 ||
                     a.lora_Lp != nullptr || a.y_amax != nullptr;
    p.num_full = p.num_tiles;
    {
        const int R = p.num_tiles % max_clusters;
        if (!epi && R > 0 && 2 * R <= max_clusters) p.num_full = p.num_tiles - R;
    }
    p.num_units = p.num_full + 2 * (p.num_tiles - p.num_full);
    p.lora_r = a.lora_Lp != nullptr ? static_cast<int>(a.lora_r) : 0;
    p.y_amax = a.y_amax;
    p.inject = debug_state().inject;
    p.timeout_ns = debug_state().timeout_ns;
    p.err = device_error_word();
    if (p.err == nullptr) return cudaErrorInvalidSymbol;
    const int clusters = p.num_units < max_clusters ? p.num_units : max_clusters;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e =
        a.y_amax != nullptr
            ? cudaLaunchKernelEx(&cfg, gemm_pair_kernel<2>, tmA, tmB, tmSA, tmSB, tmY, tmYq, tmL,
                                 tmLB, tmB64, p)
        : epi ? cudaLaunchKernelEx(&cfg, gemm_pair_kernel<1>, tmA, tmB, tmSA, tmSB, tmY, tmYq, tmL,
                                   tmLB, tmB64, p)
              : cudaLaunchKernelEx(&cfg, gemm_pair_kernel<0>, tmA, tmB, tmSA, tmSB, tmY, tmYq, tmL,
                                   tmLB, tmB64, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace nvfp4
