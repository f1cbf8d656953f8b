// Block-scaled FP4 GEMM on the sm_103a tensor cores (tcgen05, kind::mxf4nvf4).
//
//   Y[m, n] = bf16( g_a * g_b * sum_k e2m1(A[m,k]) e4m3(SA[m,k/16])
//                                     e2m1(B[n,k]) e4m3(SB[n,k/16]) )
//
// This is the "nvfp4-difusion" page's quantized matmul (section 2: two
// float4_e2m1fn_x2 operands with their E4M3 block scales, bfloat16 out),
// written for Blackwell's fifth-generation tensor cores instead of a library
// call.
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles, K in stages of
// 256 (4 MMAs of K = 64). Warp roles:
//   warp 0    TMA producer: A/B tiles (128-byte swizzle) by
//             cp.async.bulk.tensor, scale tiles (already in the 128x4 tile
//             layout) by cp.async.bulk, into a STAGES-deep ring guarded by
//             full/empty mbarriers;
//   warp 1    MMA issuer: per stage, 12 tcgen05.cp copying the stage's scales
//             shared -> TMEM, then 4 tcgen05.mma into a 128 x 256 FP32
//             accumulator in TMEM (the copies are issued by the same thread,
//             so they are ordered before the MMAs without an mbarrier
//             round trip: measured faster than a separate copy warp);
//   warp 2    allocates and frees TMEM;
//   warps 3-10 epilogue, two warps per 32-lane TMEM quarter (one per
//             128-column half): tcgen05.ld the accumulator into registers,
//             release it to the MMA warp, then scale by g_a g_b, round to
//             bfloat16 and store while the next tile's mainloop runs.
// Every tcgen05 instruction is issued from a converged warp through
// elect.sync. Every mbarrier wait is bounded in time; a wait that runs out
// records a timeout in the device error word, and all roles leave cleanly.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tensor_map.h"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;                    // FP4 elements per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK / 2;       // 16 KiB
constexpr int B_BYTES = BN * BK / 2;       // 32 KiB
constexpr int SFA_BYTES = BM * BK / 16;    // 2 KiB: 4 tiles of 512 B
constexpr int SFB_BYTES = BN * BK / 16;    // 4 KiB: 2 row groups x 4 tiles
constexpr int SF_TILE = 512;
constexpr int K_PER_MMA = 64;
constexpr int MMAS_PER_STAGE = BK / K_PER_MMA;  // 4
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;            // 256 FP32 columns
constexpr uint32_t SF_COL = 256;           // per stage: 16 (SFA) + 32 (SFB)
constexpr uint32_t SF_COLS_PER_STAGE = 48;
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 3;
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);  // 352
constexpr int GROUP_M = 16;                // tile raster: 16 M-tiles per column sweep
constexpr unsigned kAll = 0xFFFFFFFFu;

constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
constexpr int SMEM_SFA = SMEM_B + STAGES * B_BYTES;
constexpr int SMEM_SFB = SMEM_SFA + STAGES * SFA_BYTES;
constexpr int SMEM_BAR = SMEM_SFB + STAGES * SFB_BYTES;
constexpr int SMEM_USED = SMEM_BAR + 256;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // room to align the base to 1024

static_assert(STAGES * SF_COLS_PER_STAGE + SF_COL <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

struct Params {
    const uint8_t *As;   // scales of A, 128x4 tile layout
    const uint8_t *Bs;   // scales of B, 128x4 tile layout
    const float *g_a;
    const float *g_b;
    uint16_t *Y;
    int64_t ldy;
    int M, N, K;
    int num_m_tiles, num_n_tiles;
    int num_tiles;
    int y_vec;           // rows of Y start 16-byte aligned: 16-byte stores
    int inject;          // 1: the producer issues nothing (bounded-wait test)
    uint64_t timeout_ns;
    unsigned int *err;   // device error word
};

struct Shared {
    uint64_t full[STAGES];     // TMA -> MMA: stage (A, B, scales) landed
    uint64_t empty[STAGES];    // MMA -> TMA: stage consumed
    uint64_t acc_full;         // MMA -> epilogue: accumulator complete
    uint64_t acc_empty;        // epilogue -> MMA: accumulator drained
    uint64_t drain_mma;        // teardown after an abort: MMAs issued have completed
    uint32_t tmem_base;
    volatile uint32_t abort_flag;
};
static_assert(sizeof(Shared) <= 256, "barrier area");

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int &mt,
                                            int &nt) {
    const int per_group = group_m * num_n;
    const int group = t / per_group;
    const int first_m = group * group_m;
    const int gsz = min(num_m - first_m, group_m);
    const int local = t - group * per_group;
    mt = first_m + local % gsz;
    nt = local / gsz;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Bounded wait by lane 0 of a converged warp, also giving up once another
// role has aborted; the outcome is broadcast to the warp.
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

__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Shared &sh = *reinterpret_cast<Shared *>(smem + SMEM_BAR);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_k = p.K / BK;
    const int kb4 = p.K / 64;  // 512-byte scale tiles per 128-row group
    const int n_sf_groups = (p.N + 127) / 128;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.acc_full, 1);
        mbar_init(&sh.acc_empty, kEpiWarps);
        mbar_init(&sh.drain_mma, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2) {
        tmem_alloc(&sh.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    // The set-up above overlaps the previous kernel when launched as a
    // programmatic dependent; operands and scales are read only after it.
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        const uint64_t pol = policy_evict_last();
        int g = 0;  // stage counter over this CTA's tiles
        bool ok = !p.inject;
        for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
            int mt, nt;
            tile_coords(t, p.num_m_tiles, p.num_n_tiles, GROUP_M, mt, nt);
            const bool two_groups = (nt * 2 + 1) < n_sf_groups;
            const uint32_t tx = A_BYTES + B_BYTES + SFA_BYTES + (two_groups ? 2 : 1) * (SFB_BYTES / 2);
            for (int kt = 0; kt < num_k; ++kt, ++g) {
                const int s = g % STAGES;
                if (!warp_wait(&sh.empty[s], ((g / STAGES) & 1) ^ 1, p, sh)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sh.full[s], tx);
                    tma_load_2d(smem + SMEM_A + s * A_BYTES, &tmA, &sh.full[s], kt * (BK / 2),
                                mt * BM, pol);
                    tma_load_2d(smem + SMEM_B + s * B_BYTES, &tmB, &sh.full[s], kt * (BK / 2),
                                nt * BN, pol);
                    const uint8_t *sa = p.As + (static_cast<int64_t>(mt) * kb4 + kt * 4) * SF_TILE;
                    bulk_load(smem + SMEM_SFA + s * SFA_BYTES, sa, SFA_BYTES, &sh.full[s], pol);
                    // B scales: two 128-row groups of 2 KiB (the second only
                    // when the tile reaches past the first 128 rows of B)
                    const uint8_t *sb = p.Bs + (static_cast<int64_t>(nt * 2) * kb4 + kt * 4) * SF_TILE;
                    uint8_t *sdst = smem + SMEM_SFB + s * SFB_BYTES;
                    bulk_load(sdst, sb, SFB_BYTES / 2, &sh.full[s], pol);
                    if (two_groups)
                        bulk_load(sdst + SFB_BYTES / 2, sb + static_cast<int64_t>(kb4) * SF_TILE,
                                  SFB_BYTES / 2, &sh.full[s], pol);
                }
                __syncwarp();
            }
        }
        if (!ok && !p.inject && lane == 0) {
            // let copies already issued land before the CTA exits: the last
            // fill of stage s completes that stage's phase (fills - 1)
            for (int s = 0; s < STAGES && s < g; ++s) {
                const int fills = (g - s + STAGES - 1) / STAGES;
                mbar_wait(&sh.full[s], (fills - 1) & 1, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_mxf4nvf4(BM, BN);
        int g = 0, it = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++it) {
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
                // scales shared -> TMEM, issued in order ahead of the MMAs that
                // read them (same-thread tcgen05.cp -> tcgen05.mma is ordered)
                const uint32_t sf_a = tmem + SF_COL + s * SF_COLS_PER_STAGE;
                const uint32_t sf_b = sf_a + 16;
                const uint32_t sfa_smem = smem_addr(smem + SMEM_SFA + s * SFA_BYTES);
                const uint32_t sfb_smem = smem_addr(smem + SMEM_SFB + s * SFB_BYTES);
#pragma unroll
                for (int j = 0; j < MMAS_PER_STAGE; ++j) {
                    tmem_cp_32x128b_x4_elect(sf_a + j * 4, sdesc_sf(sfa_smem + j * SF_TILE));
                    tmem_cp_32x128b_x4_elect(sf_b + j * 8, sdesc_sf(sfb_smem + j * SF_TILE));
                    tmem_cp_32x128b_x4_elect(sf_b + j * 8 + 4,
                                             sdesc_sf(sfb_smem + SFB_BYTES / 2 + j * SF_TILE));
                }
                const uint32_t a_smem = smem_addr(smem + SMEM_A + s * A_BYTES);
                const uint32_t b_smem = smem_addr(smem + SMEM_B + s * B_BYTES);
#pragma unroll
                for (int j = 0; j < MMAS_PER_STAGE; ++j)
                    mma_mxf4nvf4_elect(tmem + ACC_COL, sdesc_sw128(a_smem + j * 32),
                                       sdesc_sw128(b_smem + j * 32), idesc, sf_a + j * 4,
                                       sf_b + j * 8, (kt | j) != 0);
                tc_commit_elect(&sh.empty[s]);
            }
            if (ok) tc_commit_elect(&sh.acc_full);
        }
        if (!ok) {
            // MMAs already issued must complete before TMEM is released
            tc_commit_elect(&sh.drain_mma);
            if (lane == 0) mbar_wait(&sh.drain_mma, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 2) {
        // TMEM allocator only
    } else {
        // -------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int half = (warp - kFirstEpiWarp) >> 2;  // which 128 columns
        const float alpha = __fmul_rn(*p.g_a, *p.g_b);
        int it = 0;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
            if (!warp_wait(&sh.acc_full, it & 1, p, sh)) break;
            tc_fence_after();
            int mt, nt;
            tile_coords(t, p.num_m_tiles, p.num_n_tiles, GROUP_M, mt, nt);
            const uint32_t t_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + ACC_COL +
                                    static_cast<uint32_t>(half * 128);
            uint32_t packed[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[c * 16 + i] = pack_bf16x2(__uint_as_float(r[2 * i]) * alpha,
                                                     __uint_as_float(r[2 * i + 1]) * alpha);
            }
            // accumulator drained into registers: hand it back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty);

            const int row = mt * BM + quarter * 32 + lane;
            const int n0 = nt * BN + half * 128;
            if (row < p.M) {
                uint16_t *yrow = p.Y + static_cast<int64_t>(row) * p.ldy;
                if (p.y_vec && n0 + 128 <= p.N) {
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
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

// Packed-code operand (rows x K/2 bytes) as a 2-D byte tensor, box of
// 128 bytes (256 FP4 values) x box_rows rows, 128-byte swizzle.
bool make_operand_map(CUtensorMap *map, const uint8_t *ptr, int64_t rows, int64_t K,
                      uint32_t box_rows) {
    return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, K / 2, rows, K / 2, 128u,
                       box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t st) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    static DeviceOnce once;
    static int max_ctas_of[kMaxDevices + 1] = {};
    const cudaError_t e_setup = once.run([](int slot) {
        const cudaError_t e = cudaFuncSetAttribute(
            gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e == cudaSuccess) max_ctas_of[slot] = launch_cfg().num_sms;
        return e;
    });
    if (e_setup != cudaSuccess) return e_setup;
    const int max_ctas = max_ctas_of[device_slot()];
    CUtensorMap tmA, tmB;
    if (!make_operand_map(&tmA, a.Aq, a.M, a.K, BM)) return cudaErrorInvalidValue;
    if (!make_operand_map(&tmB, a.Bq, a.N, a.K, BN)) return cudaErrorInvalidValue;
    Params p;
    p.As = a.As;
    p.Bs = a.Bs;
    p.g_a = a.g_a;
    p.g_b = a.g_b;
    p.Y = a.Y;
    p.ldy = a.ldy;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.K = static_cast<int>(a.K);
    p.num_m_tiles = static_cast<int>((a.M + BM - 1) / BM);
    p.num_n_tiles = static_cast<int>((a.N + BN - 1) / BN);
    p.num_tiles = p.num_m_tiles * p.num_n_tiles;
    p.y_vec = (a.ldy % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.Y) & 15) == 0);
    p.inject = debug_state().inject;
    p.timeout_ns = debug_state().timeout_ns;
    p.err = device_error_word();
    if (p.err == nullptr) return cudaErrorInvalidSymbol;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0] = pdl_attribute();
    cfg.gridDim = dim3(p.num_tiles < max_ctas ? p.num_tiles : max_ctas, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_kernel, tmA, tmB, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace nvfp4
