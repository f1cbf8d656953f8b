// Skinny-M block-scaled FP4 GEMM (LLM decode: M = 1 .. 128 tokens against a
// wide weight), computed as Y^T = W X^T so that the 128-row tensor-core M
// dimension is filled with weight rows and the few activation rows become
// the MMA's N dimension (64 or 128; the rows of X beyond the M that is
// loaded give output columns that are never stored):
//
//   D[n, m] = sum_k e2m1(Wq[n,k]) e4m3(Ws[n,k/16]) e2m1(Xq[m,k]) e4m3(Xs[m,k/16])
//   Y[m, n] = bf16(g_x * g_w * D[n, m])
//
// Same arithmetic as the large-M kernel (the "nvfp4-difusion" page's block-
// scaled matmul, section 2); only the roles of the operands are swapped. The
// regime is bound by streaming the weights from HBM once (N K / 2 bytes of
// codes plus N K / 16 of scales): each 128-row weight tile streams through a
// ring of stages (two 256-deep K chunks per stage when K allows; 3 to 8
// stages, as many as fit), X's chunk riding along.
//
// The weights do not depend on the kernel this one follows (the activation
// quantizer, launched as its programmatic predecessor), so the producer
// issues the first stages' weight loads before it waits for that kernel,
// and the first bytes' HBM latency overlaps the quantizer.
//
// Balance (SPLIT = 2, up to 8 activation rows): the 27648 x 5120 FFN-up
// weight is 216 tiles, one round of 148 plus a partial round of 68, in which
// 80 SMs would idle and the 68 busy ones cannot draw the HBM bandwidth that
// 148 do (measured: ~6.1 TB/s in the full round, ~4 TB/s in the partial
// one). Launched as
// clusters of two CTAs, every CTA streams whole tiles round robin, and the
// tiles of the partial last round (when they fit on half the CTAs) are
// split by K: CTA r of cluster c streams K half r of tail tile c. CTA 1
// sends its FP32 partial accumulator (128 weight rows x the loaded
// activation rows) into CTA 0's shared memory (st.shared::cluster +
// release arrive); CTA 0 adds it to its own (one IEEE addition per
// element, so the result does not depend on which half finishes first),
// scales and stores Y.
//
// FUSED (M <= kSkinnyFusedMaxM, K <= kSkinnyFusedMaxK): no codes of X ever
// reach HBM. At the start, the epilogue and quantizer warps read the
// bfloat16 X, compute g_x when it is not given (the same integer amax and
// IEEE division as nvfp4_global_scale) and quantize all of X
// (quant_math.cuh, the bytes of nvfp4_quantize) into a resident
// shared-memory copy: E2M1 codes in 128-byte-swizzled chunks and E4M3
// scales in the tensor-core tile layout. The ring then streams only
// weights. Every CTA quantizes the same small X, which overlaps the ring
// filling up while M is a few rows; beyond that, one small quantize launch
// costs less, hence the row limit.
//
// Warps: 0 TMA producer, 1 MMA issuer (per K = 64 step its two scale copies
// to TMEM and the MMA under one elect.sync), 2 TMEM allocator, 3-6
// epilogue (one per 32-lane TMEM quarter), 7-10 quantizers (FUSED only).
// All waits are bounded; a timeout is recorded and every role leaves.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "tensor_map.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace nvfp4 {

namespace {

constexpr int SK_BM = 128;                 // weight rows per tile
constexpr int SK_BK = 256;                 // K per chunk
constexpr int SK_SF_TILE = 512;
constexpr unsigned kAllLanes = 0xFFFFFFFFu;

// NX: MMA N (64 or 128); XR <= NX: rows of X loaded (or quantized);
// KC: 256-deep K chunks per pipeline stage (2 when the K range allows: two
// weight boxes per stage halve the per-stage costs of the ring);
// SPLIT: 2 = clusters of two CTAs that split the partial last round's
// tiles by K.
template <int NX, int XR, bool FUSED, int KC, int SPLIT>
struct SkCfg {
    static constexpr int W_CHUNK = SK_BM * SK_BK / 2;             // 16 KiB per K chunk
    // X chunks sit XR rows apart; the MMA reads NX >= XR rows from each, so
    // rows XR .. NX-1 of a chunk are the next chunk's (or the scales') bytes
    // and only feed output columns that are never stored
    static constexpr int X_CHUNK = XR * SK_BK / 2;
    // FUSED: resident X for K up to kSkinnyFusedMaxK
    static constexpr int RES_CHUNKS = FUSED ? static_cast<int>(kSkinnyFusedMaxK / SK_BK) : 0;
    static constexpr int XRES_BYTES = RES_CHUNKS * X_CHUNK;
    static constexpr int SFXRES_BYTES = RES_CHUNKS * 2048;       // 4 scale tiles per chunk
    // SPLIT: receive buffer of the partner's partial accumulator of a tail
    // tile (CTA 0), FP32 [activation row][weight row]
    static constexpr int NBUF = SPLIT == 1 ? 0 : 1;
    static constexpr int RECV_ONE = SK_BM * XR * 4;
    static constexpr int RECV_BYTES = NBUF * RECV_ONE;
    static constexpr int OFF_RECV = XRES_BYTES + SFXRES_BYTES;
    static constexpr int RING = OFF_RECV + RECV_BYTES;            // ring after these
    // one stage: weights (KC chunks) and their scales; unfused: X's chunks
    // and scales too
    static constexpr int W_BYTES = KC * W_CHUNK;
    static constexpr int X_BYTES = FUSED ? 0 : KC * X_CHUNK;
    static constexpr int X_LOAD = X_BYTES;                        // bytes of codes loaded
    static constexpr int SFW_BYTES = KC * 2048;
    static constexpr int SFX_BYTES = FUSED ? 0 : KC * 2048;
    static constexpr int OFF_W = 0;
    static constexpr int OFF_X = OFF_W + W_BYTES;
    static constexpr int OFF_SFW = OFF_X + X_BYTES;
    static constexpr int OFF_SFX = OFF_SFW + SFW_BYTES;
    static constexpr int STAGE_RAW = OFF_SFX + SFX_BYTES;
    static constexpr int STAGE = (STAGE_RAW + 1023) / 1024 * 1024;
    static constexpr int BUDGET = 220 * 1024;
    static constexpr int STAGES = (BUDGET - RING) / STAGE < 8 ? (BUDGET - RING) / STAGE : 8;
    static constexpr int BAR_OFF = RING + STAGES * STAGE;
    static constexpr int SMEM = BAR_OFF + 512 + 1024;
    static constexpr int EPI_WARPS = 4;
    // fused: warps that only quantize X at the start (with the epilogue
    // warps); latency-bound, so more warps quantize faster (M = 8: 4 -> 12
    // warps, 23.0 -> 21.4 us per call)
    static constexpr int Q_WARPS = FUSED ? 12 : 0;
    static constexpr int THREADS = 32 * (3 + EPI_WARPS + Q_WARPS);
    static constexpr uint32_t ACC_COL = 0;                        // NX columns
    static constexpr uint32_t SF_COL = 128;                       // per stage 16 KC (W) + 16 KC (X)
    static constexpr uint32_t SF_COLS = 32 * KC;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(!FUSED || XR == 8, "the resident X holds 8 rows");
    static_assert(SPLIT == 1 || SPLIT == 2, "one or two K ranges");
    static_assert(SF_COL + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(RING % 1024 == 0 && OFF_X % 1024 == 0 && X_CHUNK % 1024 == 0 &&
                      STAGE % 1024 == 0 && OFF_RECV % 1024 == 0,
                  "swizzled tiles need 1024-B alignment");
};

struct SkParams {
    const uint8_t *Wq;   // weight codes, N x K/2 (row-major: a tile is one contiguous range)
    const uint8_t *Ws;   // weight scales, 128x4 tile layout
    const uint8_t *Xs;   // activation scales, 128x4 tile layout (unfused)
    const uint16_t *X;   // bfloat16 activation (fused; read for amax when g_x is null)
    int64_t ldx;
    const float *g_x;    // fused: null = compute amax(|X|) / (6 * 448) in the kernel
    const float *g_w;    // one per weight group
    WeightGroups groups;
    uint16_t *Y;         // null: the bfloat16 output is not stored
    int64_t ldy;
    // epilogue extensions (see SkinnyArgs): bias, re-quantization of Y, amax of Y
    const uint16_t *bias;
    const float *g_y;
    uint8_t *Yq;
    uint8_t *Ys;
    uint32_t *y_amax;
    int M, N, K;
    int n_tiles;
    int n_tail;          // SPLIT: tiles of the partial last round split by K (the last n_tail)
    // testing hook (fused): CTA 0 copies the activation operand it quantized
    // into shared memory out to these buffers (codes M x K/2, tile-layout
    // scales with the padding rows of the first 128-row group zeroed)
    uint8_t *dbg_xq;
    uint8_t *dbg_xs;
    int inject;
    uint64_t timeout_ns;
    unsigned int *err;
};

template <int STAGES>
struct SkShared {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t xready;           // fused: the resident X is quantized
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t drain;
    uint64_t recv_full;        // SPLIT, CTA 0: the partner's partial has landed
    uint32_t tmem_base;
    volatile uint32_t abort_flag;
    float g_x;                 // fused: activation global scale used by this CTA
    uint32_t amax_part[16];    // fused: per-warp amax of X (bfloat16 bits)
};
static_assert(sizeof(SkShared<8>) <= 512, "barrier area");

// A CTA's work: whole tiles round robin over the grid, then (SPLIT) one K
// half of a tail tile. Unit u covers stages kc0 / KC .. + nk of tile nt
// (kc0 in 256-deep chunks).
struct SkUnit {
    int nt, kc0, nk;
    bool half;
};

struct SkWork {
    int n_whole;     // whole tiles of this CTA
    int nk_whole;    // stages per whole tile
    int tail;        // tail tile of this CTA's cluster, or -1
    int tail_kc0;    // its first chunk (this CTA's K half)

    __device__ __forceinline__ int units() const { return n_whole + (tail >= 0 ? 1 : 0); }
    __device__ __forceinline__ SkUnit unit(int u) const {
        if (u < n_whole)
            return {static_cast<int>(blockIdx.x + u * gridDim.x), 0, nk_whole, false};
        return {tail, tail_kc0, nk_whole / 2, true};
    }
};

template <int KC, int SPLIT>
__device__ __forceinline__ SkWork sk_work(const SkParams &p, int rank) {
    SkWork w;
    const int n_full = p.n_tiles - (SPLIT == 2 ? p.n_tail : 0);
    const int b = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    w.n_whole = b < n_full ? (n_full - b + G - 1) / G : 0;
    w.nk_whole = p.K / (SK_BK * KC);
    const int cid = b / SPLIT;
    w.tail = (SPLIT == 2 && cid < p.n_tail) ? n_full + cid : -1;
    w.tail_kc0 = rank * (p.K / SK_BK / 2);
    return w;
}

// Stage g of this CTA's work -> (tile, first 256-deep chunk); false past the end.
__device__ __forceinline__ bool sk_stage(const SkWork &w, int g, int &nt, int &k0, int kc) {
    for (int u = 0; u < w.units(); ++u) {
        const SkUnit un = w.unit(u);
        if (g < un.nk) {
            nt = un.nt;
            k0 = un.kc0 + g * kc;
            return true;
        }
        g -= un.nk;
    }
    return false;
}

template <int STAGES>
__device__ __forceinline__ bool sk_wait(uint64_t *bar, uint32_t parity, const SkParams &p,
                                        SkShared<STAGES> &sh, bool cluster_acquire = false) {
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
    ok = __shfl_sync(kAllLanes, ok, 0);
    // every lane acquires what the partner CTA released (the phase has
    // completed, so this probe returns at once)
    if (ok && cluster_acquire) (void)mbar_try_wait_cluster(smem_addr(bar), parity);
    return ok != 0;
}

// Fused path, run by the epilogue and quantizer warps (warps 3 .. 3 + 16,
// 512 threads): g_x (when not given: the same integer amax and IEEE
// division as nvfp4_global_scale, so the bytes match the unfused path),
// then all of X (rows < M; rows M .. XR-1 only feed unstored columns)
// quantized into the resident copy. Block (row r, 16-element block kb):
// codes in 256-deep chunk kb / 16 (128-byte swizzle: 16-byte piece k of
// row r at k ^ (r % 8)), scale at the tile layout's byte.
template <class C, int S>
__device__ __forceinline__ void quantize_x_resident(const SkParams &p, SkShared<S> &sh,
                                                    uint8_t *xres, uint8_t *sfxres) {
    constexpr int kWarps = C::EPI_WARPS + C::Q_WARPS;
    constexpr int kThr = 32 * kWarps;
    static_assert(kWarps <= 16, "per-warp amax slots");
    const int qt = threadIdx.x - 32 * 3;  // 0 .. kThr - 1
    const int lane = threadIdx.x & 31;
    float gx;
    if (p.g_x != nullptr) {
        gx = *p.g_x;
    } else {
        const uint32_t vpr = static_cast<uint32_t>(p.K / 8);
        const uint32_t total = static_cast<uint32_t>(p.M) * vpr;
        const uint32_t m16 = 0x7FFF7FFFu;
        uint32_t acc = 0;
        uint32_t i = qt;
        for (; i + 7 * kThr < total; i += 8 * kThr) {  // eight loads in flight
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t j = i + u * kThr;
                const uint32_t r = j / vpr, c = j - r * vpr;
                v[u] = *reinterpret_cast<const uint4 *>(p.X + r * p.ldx + c * 8ull);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                acc = max_u16x2(acc, max_u16x2(max_u16x2(v[u].x & m16, v[u].y & m16),
                                               max_u16x2(v[u].z & m16, v[u].w & m16)));
        }
        for (; i < total; i += kThr) {
            const uint32_t r = i / vpr, c = i - r * vpr;
            const uint4 v = *reinterpret_cast<const uint4 *>(p.X + r * p.ldx + c * 8ull);
            acc = max_u16x2(acc, max_u16x2(max_u16x2(v.x & m16, v.y & m16),
                                           max_u16x2(v.z & m16, v.w & m16)));
        }
        uint32_t a = max(acc & 0xFFFFu, acc >> 16);
        a = __reduce_max_sync(kAllLanes, a);
        if (lane == 0) sh.amax_part[qt >> 5] = a;
        asm volatile("bar.sync 1, %0;" ::"n"(kThr) : "memory");
        a = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) a = max(a, sh.amax_part[w]);
        const float amax = __uint_as_float(a << 16);
        gx = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
    }
    if (qt == 0) sh.g_x = gx;
    const int kbpr = p.K / 16;
    const int nblk = p.M * kbpr;
    constexpr int U = 4;  // blocks per thread per round, loads issued first
    for (int b0 = qt; b0 < nblk; b0 += U * kThr) {
        uint4 v0[U], v1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * kThr;
            v0[u] = make_uint4(0, 0, 0, 0);
            v1[u] = v0[u];
            if (b < nblk) {
                const int r = b / kbpr, kb = b - r * kbpr;
                const uint4 *src = reinterpret_cast<const uint4 *>(p.X + r * p.ldx + kb * 16ll);
                v0[u] = src[0];
                v1[u] = src[1];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * kThr;
            if (b >= nblk) break;
            const int r = b / kbpr, kb = b - r * kbpr;
            uint32_t lo, hi;
            const uint32_t Sb = quantize16(v0[u], v1[u], gx, lo, hi);
            const int chunk = kb >> 4, kbc = kb & 15, piece = kbc >> 1;
            const int xoff = chunk * C::X_CHUNK + r * 128 + ((piece ^ (r & 7)) << 4) + (kbc & 1) * 8;
            const int soff = (kb >> 2) * SK_SF_TILE + (r & 31) * 16 + (r >> 5) * 4 + (kb & 3);
            if (NVFP4_CHECK(xoff + 8 <= C::XRES_BYTES && r * 128 < C::X_CHUNK))
                *reinterpret_cast<uint2 *>(xres + xoff) = make_uint2(lo, hi);
            if (NVFP4_CHECK(soff < C::SFXRES_BYTES)) sfxres[soff] = static_cast<uint8_t>(Sb);
        }
    }
    fence_proxy_async_shared();  // generic-proxy writes -> tensor core reads
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.xready);
    __syncwarp();
}

// The decode epilogue with the extensions (bias, re-quantization of Y,
// amax of Y) for one weight row n = lane's row of the tile (lane = weight
// row, column m = activation row, as the accumulator lies in TMEM), the
// arithmetic of the CTA-pair epilogue and of the standalone quantizer:
//   y = bf16(acc * alpha [+ bias[n]])  (fp32, one rounding)
// A block of 16 consecutive n is 16 lanes of the warp: its amax is a
// shuffle reduction, every lane takes the same scale byte S and multiplier,
// the even lane of each pair converts the pair, and the group's first lane
// gathers the 8 code bytes and stores them with S (tile layout; rows M ..
// 127 of the 128-row group get scale 0). Requires N % 256 == 0 with Yq,
// so every lane's n is a column of Y.
template <int XR, int NX>
__device__ __forceinline__ void sk_epilogue_ext(const SkParams &p, const float (&acc)[NX],
                                                float alpha, int n, int n_warp, int lane) {
    const bool has_bias = p.bias != nullptr;
    const bool rq = p.Yq != nullptr;
    const bool in = n < p.N;
    const float bv =
        has_bias && in ? __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16) : 0.0f;
    const float gy = rq ? *p.g_y : 1.0f;
    const int gbase = lane & 16;                  // first lane of this lane's 16-lane group
    const int n_blk = n_warp + gbase;             // first column of the group's block
    const int kb = n_blk >> 4;
    const int kb4 = p.N / 64;
    [[maybe_unused]] const uint64_t sf_end = static_cast<uint64_t>((p.M + 127) / 128) * 128 * (p.N / 16);
    uint32_t am = 0;
#pragma unroll
    for (int m = 0; m < XR; ++m) {
        if (m >= p.M) break;  // the same for every lane
        const float y = has_bias ? __fadd_rn(__fmul_rn(acc[m], alpha), bv) : acc[m] * alpha;
        const __nv_bfloat16 v = __float2bfloat16_rn(y);
        const uint32_t yb = *reinterpret_cast<const uint16_t *>(&v);
        if (p.Y != nullptr && in) p.Y[static_cast<int64_t>(m) * p.ldy + n] = static_cast<uint16_t>(yb);
        if (in) am = max(am, yb & 0x7FFFu);
        if (rq) {
            uint32_t a = yb & 0x7FFFu;
            a = max(a, __shfl_xor_sync(kAllLanes, a, 1));
            a = max(a, __shfl_xor_sync(kAllLanes, a, 2));
            a = max(a, __shfl_xor_sync(kAllLanes, a, 4));
            a = max(a, __shfl_xor_sync(kAllLanes, a, 8));
            const float amax = __uint_as_float(a << 16);
            const uint32_t S = cvt_e4m3_satfinite(__fdiv_rn(__fdiv_rn(amax, 6.0f), gy));
            const float r = scale_recip(S, gy);
            const uint64_t rr =
                (static_cast<uint64_t>(__float_as_uint(r)) << 32) | __float_as_uint(r);
            const uint32_t partner = __shfl_xor_sync(kAllLanes, yb, 1);
            const uint32_t byte = codes2(yb | (partner << 16), rr);  // valid on even lanes
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo |= (__shfl_sync(kAllLanes, byte, gbase + 2 * j) & 0xFFu) << (8 * j);
                hi |= (__shfl_sync(kAllLanes, byte, gbase + 8 + 2 * j) & 0xFFu) << (8 * j);
            }
            if ((lane & 15) == 0) {
                const int64_t qoff = static_cast<int64_t>(m) * (p.N / 2) + n_blk / 2;
                if (NVFP4_CHECK(qoff + 8 <= static_cast<int64_t>(p.M) * (p.N / 2)))
                    *reinterpret_cast<uint2 *>(p.Yq + qoff) = make_uint2(lo, hi);
                const uint64_t off = ((static_cast<uint64_t>(m >> 7) * kb4 + (kb >> 2)) << 9) +
                                     ((m & 31) << 4) + (((m & 127) >> 5) << 2) + (kb & 3);
                if (NVFP4_CHECK(off < sf_end)) p.Ys[off] = static_cast<uint8_t>(S);
            }
        }
    }
    if (rq) {
        // padding rows of the 128-row group: scale 0 for this warp's two
        // blocks, the (row, block) pairs spread over the 32 lanes
        const int rows_pad = (p.M + 127) / 128 * 128;
        const int kb0 = n_warp >> 4;
        for (int i = lane; i < 2 * (rows_pad - p.M); i += 32) {
            const int m = p.M + (i >> 1), k = kb0 + (i & 1);
            const uint64_t off = ((static_cast<uint64_t>(m >> 7) * kb4 + (k >> 2)) << 9) +
                                 ((m & 31) << 4) + (((m & 127) >> 5) << 2) + (k & 3);
            if (NVFP4_CHECK(off < sf_end)) p.Ys[off] = 0;
        }
    }
    if (p.y_amax != nullptr) {
        am = __reduce_max_sync(kAllLanes, am);
        if (lane == 0 && am != 0u) atomicMax(p.y_amax, am);
    }
}

template <int NX, int XR, bool FUSED, int KC, int SPLIT>
__global__ void __launch_bounds__(SkCfg<NX, XR, FUSED, KC, SPLIT>::THREADS, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                  const SkParams p) {
    using C = SkCfg<NX, XR, FUSED, KC, SPLIT>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem_base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *smem = smem_base + C::RING;      // the stage ring
    uint8_t *xres = smem_base;                // fused: resident X codes
    uint8_t *sfxres = smem_base + C::XRES_BYTES;  // fused: resident X scales
    float *recv = reinterpret_cast<float *>(smem_base + C::OFF_RECV);  // SPLIT, CTA 0
    SkShared<S> &sh = *reinterpret_cast<SkShared<S> *>(smem_base + C::BAR_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = SPLIT == 2 ? static_cast<int>(cluster_ctarank()) : 0;
    const SkWork work = sk_work<KC, SPLIT>(p, rank);
    const int kb4 = p.K / 64;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.xready, C::Q_WARPS > 0 ? C::Q_WARPS + C::EPI_WARPS : 1);
        mbar_init(&sh.acc_full, 1);
        mbar_init(&sh.acc_empty, C::EPI_WARPS);
        mbar_init(&sh.drain, 1);
        mbar_init(&sh.recv_full, 32 * C::EPI_WARPS);  // every lane of CTA 1's epilogue
        sh.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmW);
        if (!FUSED) tma_prefetch_desc(&tmX);
    }
    if (warp == 2) {
        tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if (SPLIT == 2) cluster_sync_all();  // the partner's barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    // the next kernel may start its own set-up; every role that reads what
    // the previous kernel wrote (X, its codes and scales, g_x) or writes Y
    // waits for that kernel first (pdl_wait)
    pdl_launch_dependents();

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        const uint64_t pol_w = policy_evict_first();  // weights stream through once
        const uint64_t pol_x = policy_evict_last();   // X is re-read by every CTA
        constexpr uint32_t tx = C::W_BYTES + C::SFW_BYTES + C::X_LOAD + C::SFX_BYTES;
        int total = 0;
        for (int u = 0; u < work.units(); ++u) total += work.unit(u).nk;
        const bool issue = !p.inject;
        auto load_w = [&](int s, int nt, int k0) {
            uint8_t *st = smem + s * C::STAGE;
#pragma unroll
            for (int c = 0; c < KC; ++c)
                tma_load_2d(st + C::OFF_W + c * C::W_CHUNK, &tmW, &sh.full[s],
                            (k0 + c) * (SK_BK / 2), nt * SK_BM, pol_w);
            bulk_load(st + C::OFF_SFW, p.Ws + (static_cast<int64_t>(nt) * kb4 + k0 * 4) * SK_SF_TILE,
                      C::SFW_BYTES, &sh.full[s], pol_w);
        };
        auto load_x = [&](int s, int k0) {
            uint8_t *st = smem + s * C::STAGE;
#pragma unroll
            for (int c = 0; c < KC; ++c)
                tma_load_2d(st + C::OFF_X + c * C::X_CHUNK, &tmX, &sh.full[s],
                            (k0 + c) * (SK_BK / 2), 0, pol_x);
            bulk_load(st + C::OFF_SFX, p.Xs + static_cast<int64_t>(k0) * 4 * SK_SF_TILE,
                      C::SFX_BYTES, &sh.full[s], pol_x);
        };
        // the first S stages' weights before waiting for the previous kernel
        // (the slots are fresh), X's codes and scales after
        const int pre = issue ? (total < S ? total : S) : 0;
        if (lane == 0) {
            for (int g = 0; g < pre; ++g) {
                int nt, k0;
                sk_stage(work, g, nt, k0, KC);
                mbar_arrive_expect_tx(&sh.full[g], tx);
                load_w(g, nt, k0);
            }
            // Then every weight byte of this CTA's units into L2: the ring
            // holds only S stages, and until the previous kernel completes
            // (and X is known) no slot is freed; the prefetch keeps HBM busy
            // across that boundary. A tile's codes (128 rows x K/2) and its
            // scales are contiguous ranges; a split tile's is fetched by the
            // cluster's CTA 0. The weights are inputs no kernel writes, so
            // they may be read before the wait.
            if (issue) {
                for (int u = 0; u < work.units(); ++u) {
                    const SkUnit un = work.unit(u);
                    if (un.half && rank != 0) continue;
                    const int64_t row0 = static_cast<int64_t>(un.nt) * SK_BM;
                    const int64_t rows = p.N - row0 < SK_BM ? p.N - row0 : SK_BM;
                    bulk_prefetch_l2(p.Wq + row0 * (p.K / 2),
                                     static_cast<uint32_t>(rows * (p.K / 2)));
                    bulk_prefetch_l2(p.Ws + static_cast<int64_t>(un.nt) * kb4 * SK_SF_TILE,
                                     static_cast<uint32_t>(kb4 * SK_SF_TILE));
                }
            }
        }
        __syncwarp();
        pdl_wait();
        if (!FUSED && lane == 0) {
            for (int g = 0; g < pre; ++g) {
                int nt, k0;
                sk_stage(work, g, nt, k0, KC);
                load_x(g, k0);
            }
        }
        __syncwarp();
        int g = pre;
        bool ok = issue;
        for (; ok && g < total; ++g) {
            const int s = g % S;
            if (!sk_wait<S>(&sh.empty[s], ((g / S) & 1) ^ 1, p, sh)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                int nt, k0;
                sk_stage(work, g, nt, k0, KC);
                mbar_arrive_expect_tx(&sh.full[s], tx);
                load_w(s, nt, k0);
                if (!FUSED) load_x(s, k0);
            }
            __syncwarp();
        }
        if (!ok && issue && lane == 0) {
            // let the loads already issued land before the CTA exits
            for (int s = 0; s < S && s < g; ++s) {
                const int fills = (g - s + S - 1) / S;
                mbar_wait(&sh.full[s], (fills - 1) & 1, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // (reads only shared memory and TMEM, gated by the full barriers)
        constexpr uint32_t idesc = idesc_mxf4nvf4(SK_BM, NX);
        int g = 0;
        bool ok = !FUSED || sk_wait<S>(&sh.xready, 0, p, sh);
        for (int u = 0; ok && u < work.units(); ++u) {
            const SkUnit un = work.unit(u);
            if (!sk_wait<S>(&sh.acc_empty, (u & 1) ^ 1, p, sh)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kt = 0; kt < un.nk; ++kt, ++g) {
                const int s = g % S;
                if (!sk_wait<S>(&sh.full[s], (g / S) & 1, p, sh)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t *st = smem + s * C::STAGE;
                const uint32_t sf_w = tmem + C::SF_COL + s * C::SF_COLS;
                const uint32_t sf_x = sf_w + 16 * KC;
                const uint32_t sfw_smem = smem_addr(st + C::OFF_SFW);
                const uint32_t w_smem = smem_addr(st + C::OFF_W);
                // X and its scales: this stage's chunks, or (fused) the
                // resident chunks of the stage's K range
                const int xc = un.kc0 + kt * KC;
                const uint32_t x_smem = FUSED ? smem_addr(xres + xc * C::X_CHUNK)
                                              : smem_addr(st + C::OFF_X);
                const uint32_t sfx_smem = FUSED ? smem_addr(sfxres + xc * 2048)
                                                : smem_addr(st + C::OFF_SFX);
                // per K = 64 step: its two scale tiles, then the MMA, one elect
#pragma unroll
                for (int q = 0; q < 4 * KC; ++q) {
                    const int c = q >> 2, j = q & 3;  // chunk, K = 64 step within it
                    sf_copy2_mma_elect(tmem + C::ACC_COL,
                                       sdesc_sw128(w_smem + c * C::W_CHUNK + j * 32),
                                       sdesc_sw128(x_smem + c * C::X_CHUNK + j * 32), idesc,
                                       sf_w + q * 4, sf_x + q * 4, (kt | q) != 0,
                                       sdesc_sf(sfw_smem + q * SK_SF_TILE),
                                       sdesc_sf(sfx_smem + q * SK_SF_TILE));
                }
                tc_commit_elect(&sh.empty[s]);
            }
            if (ok) tc_commit_elect(&sh.acc_full);
        }
        if (!ok) {
            tc_commit_elect(&sh.drain);
            if (lane == 0) mbar_wait(&sh.drain, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 2) {
        // TMEM allocator only
    } else if (warp < 3 + C::EPI_WARPS) {
        pdl_wait();  // g_x and X come from the previous kernel; Y may be its input
        // fused: the epilogue warps first help quantize X (idle until the
        // first accumulator is complete anyway)
        if (FUSED) quantize_x_resident<C, S>(p, sh, xres, sfxres);
        if (FUSED && p.dbg_xq != nullptr && blockIdx.x == 0 && warp == 3 &&
            sk_wait<S>(&sh.xready, 0, p, sh)) {
            // testing hook: the resident operand, un-swizzled, to global
            const int kbpr = p.K / 16;
            for (int b = lane; b < p.M * kbpr; b += 32) {
                const int r = b / kbpr, kb = b - r * kbpr;
                const int chunk = kb >> 4, kbc = kb & 15, piece = kbc >> 1;
                *reinterpret_cast<uint2 *>(p.dbg_xq + static_cast<int64_t>(r) * (p.K / 2) +
                                           kb * 8) =
                    *reinterpret_cast<const uint2 *>(xres + chunk * C::X_CHUNK + r * 128 +
                                                     ((piece ^ (r & 7)) << 4) + (kbc & 1) * 8);
            }
            for (int i = lane; i < 128 * kbpr; i += 32) {
                const int r = i / kbpr, kb = i - r * kbpr;
                const int off = (kb >> 2) * SK_SF_TILE + (r & 31) * 16 + (r >> 5) * 4 + (kb & 3);
                p.dbg_xs[off] = r < p.M ? sfxres[off] : 0;
            }
            __syncwarp();
        }
        // -------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // weight row within the tile
        for (int u = 0; u < work.units(); ++u) {
            const SkUnit un = work.unit(u);
            if (!sk_wait<S>(&sh.acc_full, u & 1, p, sh)) break;
            tc_fence_after();
            const uint32_t t_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + C::ACC_COL;
            // D[n, m]: lane = weight row n, column = activation row m
            float acc[NX];
#pragma unroll
            for (int c = 0; c < NX / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[c * 32 + i] = __uint_as_float(r[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty);
            if (SPLIT == 2 && un.half) {
                // a tail tile: CTA 1 hands its K half's partial to CTA 0
                // ([m][row] in CTA 0's buffer; the buffer is used once)
                if (rank == 1) {
                    const uint32_t dst = mapa_shared(smem_addr(recv + row), 0);
#pragma unroll
                    for (int m = 0; m < XR; ++m)
                        if (NVFP4_CHECK((m * SK_BM + row + 1) * 4 <= C::RECV_BYTES))
                            st_cluster_u32(dst + m * SK_BM * 4, __float_as_uint(acc[m]));
                    mbar_arrive_cluster(mapa_shared(smem_addr(&sh.recv_full), 0));
                    continue;
                }
                if (!sk_wait<S>(&sh.recv_full, 0, p, sh, true)) break;
#pragma unroll
                for (int m = 0; m < XR; ++m)
                    if (NVFP4_CHECK((m * SK_BM + row + 1) * 4 <= C::RECV_BYTES))
                        acc[m] = __fadd_rn(acc[m], recv[m * SK_BM + row]);
            }
            // fused: the quantizer warps published g_x in shared memory before
            // the MMAs this accumulator completion follows
            const float gx = FUSED ? sh.g_x : *p.g_x;
            const float alpha = __fmul_rn(gx, p.g_w[weight_group_of(p.groups, un.nt * SK_BM)]);
            const int n = un.nt * SK_BM + row;
            const bool ext = p.bias != nullptr || p.Yq != nullptr || p.y_amax != nullptr;
            if (!ext) {
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < XR; ++m) {
                        if (m < p.M) {
                            const __nv_bfloat16 v = __float2bfloat16_rn(acc[m] * alpha);
                            p.Y[static_cast<int64_t>(m) * p.ldy + n] =
                                *reinterpret_cast<const uint16_t *>(&v);
                        }
                    }
                }
            } else if constexpr (NX <= 64) {
                // (the 128-row variant carries no extensions: the host sends
                // them only with M <= 64)
                sk_epilogue_ext<XR, NX>(p, acc, alpha, n, un.nt * SK_BM + quarter * 32, lane);
            }
        }
        __syncwarp();
    } else if (FUSED) {
        pdl_wait();
        quantize_x_resident<C, S>(p, sh, xres, sfxres);
    }

    tc_fence_before();
    __syncthreads();
    if (SPLIT == 2) cluster_sync_all();  // neither CTA leaves while the other may address it
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Tiles of the partial last round that a cluster launch splits by K: all of
// them when they fit on half the SMs, else none.
int tail_tiles(int64_t n_tiles) {
    const int64_t G = launch_cfg().num_sms & ~1;
    const int64_t rem = n_tiles % G;
    return (rem > 0 && 2 * rem <= G) ? static_cast<int>(rem) : 0;
}

template <int NX, int XR, bool FUSED, int KC, int SPLIT>
cudaError_t launch_sk(const SkinnyArgs &a, cudaStream_t st) {
    using C = SkCfg<NX, XR, FUSED, KC, SPLIT>;
    static DeviceOnce once;
    const cudaError_t e_setup = once.run([](int) {
        return cudaFuncSetAttribute(skinny_kernel<NX, XR, FUSED, KC, SPLIT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (e_setup != cudaSuccess) return e_setup;
    CUtensorMap tmW, tmX;
    if (!make_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wq, a.K / 2, a.N, a.K / 2, 128, SK_BM,
                CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (FUSED) {
        memset(&tmX, 0, sizeof(tmX));  // X is read by the quantizer warps directly
    } else {
        if (!make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Xq, a.K / 2, a.M, a.K / 2, 128, XR,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    SkParams p;
    p.Wq = a.Wq;
    p.Ws = a.Ws;
    p.Xs = a.Xs;
    p.X = a.X;
    p.ldx = a.ldx;
    p.g_x = a.g_x;
    p.g_w = a.g_w;
    p.groups = a.groups;
    p.Y = a.Y;
    p.ldy = a.ldy;
    p.bias = a.bias;
    p.g_y = a.g_y;
    p.Yq = a.Yq;
    p.Ys = a.Ys;
    p.y_amax = a.y_amax;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.K = static_cast<int>(a.K);
    p.n_tiles = static_cast<int>((a.N + SK_BM - 1) / SK_BM);
    p.n_tail = SPLIT == 2 ? tail_tiles(p.n_tiles) : 0;
    p.dbg_xq = FUSED ? a.dbg_xq : nullptr;
    p.dbg_xs = FUSED ? a.dbg_xs : nullptr;
    p.inject = debug_state().inject;
    p.timeout_ns = debug_state().timeout_ns;
    p.err = device_error_word();
    if (p.err == nullptr) return cudaErrorInvalidSymbol;
    // whole tiles round robin over the grid; with SPLIT, one cluster per
    // tail tile as well
    const int G = launch_cfg().num_sms & ~(SPLIT - 1);
    const int n_full = p.n_tiles - p.n_tail;
    int ctas = n_full < G ? n_full : G;
    if (2 * p.n_tail > ctas) ctas = 2 * p.n_tail;
    ctas = (ctas + SPLIT - 1) / SPLIT * SPLIT;
    cudaLaunchAttribute attrs[2];
    attrs[0] = pdl_attribute();
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = SPLIT;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = attrs;
    cfg.numAttrs = SPLIT == 2 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, skinny_kernel<NX, XR, FUSED, KC, SPLIT>, tmW, tmX, p);
}

// Unfused: the activation rows loaded (XR) follow M.
template <int KC, int SPLIT>
cudaError_t launch_unfused(const SkinnyArgs &a, cudaStream_t st) {
    if (a.M <= 32) return launch_sk<64, 32, false, KC, SPLIT>(a, st);
    return launch_sk<64, 64, false, KC, SPLIT>(a, st);
}

}  // namespace

cudaError_t launch_gemm_skinny(const SkinnyArgs &a, cudaStream_t st) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    if (a.M > kSkinnyMaxM) return cudaErrorInvalidValue;
    // the epilogue extensions live in the variants up to 64 activation rows
    const bool ext = a.bias != nullptr || a.Yq != nullptr || a.y_amax != nullptr;
    if (ext && (a.M > kSkinnyExtMaxM || a.fused)) return cudaErrorInvalidValue;
    // a tail to split, whose K halves are whole stages of two chunks. Only
    // for up to 8 activation rows: measured on the 27648 x 5120 weight, the
    // split saves 1.2 us at M = 1 and 2.7 us at M = 8 but costs 2.5 us at
    // M = 16 and 32, where a full-grid quantizer precedes the GEMM and the
    // cluster launch waits for it
    const bool split = a.M <= 8 && a.K % 1024 == 0 && tail_tiles((a.N + SK_BM - 1) / SK_BM) > 0;
    if (a.fused) {
        if (a.M > kSkinnyFusedMaxM || a.K > kSkinnyFusedMaxK) return cudaErrorInvalidValue;
        if (split) return launch_sk<64, 8, true, 2, 2>(a, st);
        return a.K % 512 == 0 ? launch_sk<64, 8, true, 2, 1>(a, st)
                              : launch_sk<64, 8, true, 1, 1>(a, st);
    }
    if (a.M > 64) {
        // 128 activation rows: a receive buffer would crowd out the ring
        return a.K % 512 == 0 ? launch_sk<128, 128, false, 2, 1>(a, st)
                              : launch_sk<128, 128, false, 1, 1>(a, st);
    }
    if (split) return launch_unfused<2, 2>(a, st);
    return a.K % 512 == 0 ? launch_unfused<2, 1>(a, st) : launch_unfused<1, 1>(a, st);
}

}  // namespace nvfp4
