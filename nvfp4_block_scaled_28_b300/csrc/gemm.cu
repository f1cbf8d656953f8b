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
// Structure of one CTA (one 128 x 256 output tile, K in steps of 256):
//   warp 0   TMA producer: A/B tiles (128-byte swizzle) by cp.async.bulk.tensor,
//            scale tiles (already in the 128x4 tile layout) by cp.async.bulk,
//            into a STAGES-deep ring guarded by full/empty mbarriers;
//   warp 1   allocates TMEM, then one lane copies each stage's scales
//            shared->TMEM (tcgen05.cp) and issues 4 tcgen05.mma (K = 64
//            each) accumulating into a 128 x 256 FP32 TMEM tile;
//   warps 2-5 epilogue: tcgen05.ld the accumulator (each warp owns its
//            32-lane TMEM quarter), scale by g_a * g_b, round to bfloat16
//            and store.
// Every mbarrier wait is bounded in time; a wait that runs out records a
// timeout in the device error word and the CTA leaves cleanly.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
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
constexpr int kThreads = 192;
constexpr int GROUP_M = 16;                // tile raster: 16 M-tiles per column sweep

constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
constexpr int SMEM_SFA = SMEM_B + STAGES * B_BYTES;
constexpr int SMEM_SFB = SMEM_SFA + STAGES * SFA_BYTES;
constexpr int SMEM_BAR = SMEM_SFB + STAGES * SFB_BYTES;
constexpr int SMEM_USED = SMEM_BAR + 256;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // room to align the base to 1024

static_assert(STAGES * (SF_COLS_PER_STAGE) + SF_COL <= TMEM_COLS, "TMEM budget");
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
    int y_vec;           // rows of Y start 16-byte aligned: 16-byte stores
    int inject;          // 1: the producer issues nothing (bounded-wait test)
    uint64_t timeout_ns;
    unsigned int *err;   // device error word
};

struct Shared {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full;
    uint32_t tmem_base;
    volatile uint32_t abort_flag;
};

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int &mt, int &nt) {
    const int per_group = GROUP_M * num_n;
    const int group = t / per_group;
    const int first_m = group * GROUP_M;
    const int gsz = min(num_m - first_m, GROUP_M);
    const int local = t - group * per_group;
    mt = first_m + local % gsz;
    nt = local / gsz;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
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
    int mt, nt;
    tile_coords(blockIdx.x, p.num_m_tiles, p.num_n_tiles, mt, nt);
    const int m0 = mt * BM, n0 = nt * BN;
    const int num_k = p.K / BK;
    const int kb4 = p.K / 64;  // 512-byte scale tiles per 128-row group
    const int n_sf_groups = (p.N + 127) / 128;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.acc_full, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    // Roles run warp-wide loops in which lane 0 waits and issues; the other
    // lanes follow through __shfl_sync, so every warp reaches the final
    // barrier and the .sync.aligned tcgen05 instructions converged.
    constexpr unsigned kAll = 0xFFFFFFFFu;
    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        const uint64_t pol = policy_evict_last();
        const bool two_groups = (nt * 2 + 1) < n_sf_groups;
        const uint32_t tx = A_BYTES + B_BYTES + SFA_BYTES + (two_groups ? 2 : 1) * (SFB_BYTES / 2);
        int issued_total = 0;
        bool ok = true;
        for (int kt = 0; kt < num_k && !p.inject; ++kt) {
            const int s = kt % STAGES;
            const uint32_t ph = (kt / STAGES) & 1;
            int go = 1;
            if (lane == 0) {
                if (!mbar_wait(&sh.empty[s], ph ^ 1, p.timeout_ns)) {
                    record_timeout(p.err);
                    sh.abort_flag = 1;
                    go = 0;
                } else if (sh.abort_flag) {
                    go = 0;
                } else {
                    mbar_arrive_expect_tx(&sh.full[s], tx);
                    tma_load_2d(smem + SMEM_A + s * A_BYTES, &tmA, &sh.full[s], kt * (BK / 2), m0,
                                pol);
                    tma_load_2d(smem + SMEM_B + s * B_BYTES, &tmB, &sh.full[s], kt * (BK / 2), n0,
                                pol);
                    const uint8_t *sa = p.As + (static_cast<int64_t>(mt) * kb4 + kt * 4) * SF_TILE;
                    bulk_load(smem + SMEM_SFA + s * SFA_BYTES, sa, SFA_BYTES, &sh.full[s], pol);
                    const uint8_t *sb =
                        p.Bs + (static_cast<int64_t>(nt * 2) * kb4 + kt * 4) * SF_TILE;
                    bulk_load(smem + SMEM_SFB + s * SFB_BYTES, sb, SFB_BYTES / 2, &sh.full[s], pol);
                    if (two_groups)
                        bulk_load(smem + SMEM_SFB + s * SFB_BYTES + SFB_BYTES / 2,
                                  sb + static_cast<int64_t>(kb4) * SF_TILE, SFB_BYTES / 2,
                                  &sh.full[s], pol);
                }
            }
            go = __shfl_sync(kAll, go, 0);
            if (!go) {
                ok = false;
                break;
            }
            ++issued_total;
        }
        if (!ok && lane == 0) {
            // let the copies already issued land before the CTA exits: the
            // last fill of stage s completes phase (fills_of_s - 1)
            for (int s = 0; s < STAGES && s < issued_total; ++s) {
                const int fills = (issued_total - s + STAGES - 1) / STAGES;
                mbar_wait(&sh.full[s], (fills - 1) & 1, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_mxf4nvf4(BM, BN);
        for (int kt = 0; kt < num_k; ++kt) {
            const int s = kt % STAGES;
            const uint32_t ph = (kt / STAGES) & 1;
            int go = 1;
            if (lane == 0) {
                if (!mbar_wait(&sh.full[s], ph, p.timeout_ns)) {
                    record_timeout(p.err);
                    sh.abort_flag = 1;
                    go = 0;
                } else {
                    tc_fence_after();
                    const uint32_t sf_a = tmem + SF_COL + s * SF_COLS_PER_STAGE;
                    const uint32_t sf_b = sf_a + 16;
                    const uint32_t sfa_smem = smem_addr(smem + SMEM_SFA + s * SFA_BYTES);
                    const uint32_t sfb_smem = smem_addr(smem + SMEM_SFB + s * SFB_BYTES);
#pragma unroll
                    for (int j = 0; j < MMAS_PER_STAGE; ++j) {
                        tmem_cp_32x128b_x4(sf_a + j * 4, sdesc_sf(sfa_smem + j * SF_TILE));
                        tmem_cp_32x128b_x4(sf_b + j * 8, sdesc_sf(sfb_smem + j * SF_TILE));
                        tmem_cp_32x128b_x4(sf_b + j * 8 + 4,
                                           sdesc_sf(sfb_smem + SFB_BYTES / 2 + j * SF_TILE));
                    }
                    const uint32_t a_smem = smem_addr(smem + SMEM_A + s * A_BYTES);
                    const uint32_t b_smem = smem_addr(smem + SMEM_B + s * B_BYTES);
#pragma unroll
                    for (int j = 0; j < MMAS_PER_STAGE; ++j)
                        mma_mxf4nvf4(tmem + ACC_COL, sdesc_sw128(a_smem + j * 32),
                                     sdesc_sw128(b_smem + j * 32), idesc, sf_a + j * 4,
                                     sf_b + j * 8, (kt | j) != 0);
                    tc_commit(&sh.empty[s]);
                }
            }
            go = __shfl_sync(kAll, go, 0);
            if (!go) break;
        }
        if (lane == 0) {
            __threadfence_block();
            tc_commit(&sh.acc_full);  // arrives once every MMA issued above has completed
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        int ok = mbar_wait(&sh.acc_full, 0, p.timeout_ns) ? 1 : 0;
        ok = __all_sync(kAll, ok);
        if (!ok && lane == 0) record_timeout(p.err);
        tc_fence_after();
        ok = __shfl_sync(kAll, ok && !sh.abort_flag, 0);
        if (ok) {
            const float alpha = __fmul_rn(*p.g_a, *p.g_b);
            const int row = m0 + quarter * 32 + lane;
            const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + ACC_COL;
            uint16_t *yrow = p.Y + static_cast<int64_t>(row) * p.ldy;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + c * 32, r);
                tmem_ld_wait();
                const int n = n0 + c * 32;
                if (row < p.M && n < p.N) {
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        packed[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * alpha,
                                                __uint_as_float(r[2 * i + 1]) * alpha);
                    if (n + 32 <= p.N && p.y_vec) {
                        uint4 *dst = reinterpret_cast<uint4 *>(yrow + n);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                                packed[4 * i + 3]);
                    } else {
                        for (int i = 0; i < 32 && n + i < p.N; ++i)
                            yrow[n + i] = static_cast<uint16_t>(
                                (packed[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu);
                    }
                }
                __syncwarp();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// Packed-code operand (rows x K/2 bytes) as a 2-D byte tensor, box of
// 128 bytes (256 FP4 values) x box_rows rows, 128-byte swizzle.
bool make_operand_map(CUtensorMap *map, const uint8_t *ptr, int64_t rows, int64_t K,
                      uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    cuuint32_t box[2] = {128u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t st) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
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
    p.y_vec = (a.ldy % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.Y) & 15) == 0);
    p.inject = debug_state().inject;
    p.timeout_ns = debug_state().timeout_ns;
    p.err = device_error_word();
    if (p.err == nullptr) return cudaErrorInvalidSymbol;
    const int tiles = p.num_m_tiles * p.num_n_tiles;
    gemm_kernel<<<tiles, kThreads, SMEM_ALLOC, st>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace nvfp4
