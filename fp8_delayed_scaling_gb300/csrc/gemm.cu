// gemm.cu — FP8 GEMM on the tcgen05 tensor cores with a dequantising epilogue.
//
// "FP8 低精度训练：Transformer Engine 简析", §三.3: fp8_gemm multiplies the FP8
// casts, reading the scales kept in fp8_meta; §三.4: FP8 math runs only on the
// tensor cores, two FP8 matrices in and a high-precision (FP16/FP32) result out,
// and every GEMM dimension is a multiple of 16.  The page's kernel unit
// (wmma::mma_sync, 16x16) is the Hopper-era interface; on sm_103a the same
// contraction is a tcgen05.mma of kind::f8f6f4 (M=128, N=256, K=32 per
// instruction) with the accumulator in tensor memory.
//
//   D[m,n] = round( acc[m,n] * fl32(a_scale_inv * b_scale_inv) + bias[n] ),
//   acc = sum_k A[m,k] * B[n,k] (fp32 accumulate), A [M x K], B [N x K].
//
// Kernel structure (persistent, one CTA per SM, 192 threads):
//   warp 0      TMA producer: 128x128-byte A and 256x128-byte B tiles into a
//               STAGES-deep ring of 128-byte-swizzled shared-memory stages.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//               issues 4 MMAs per stage from one thread; tcgen05.commit frees
//               the stage and, after the last k-block, hands the accumulator
//               to the epilogue.
//   warps 2-5   epilogue: tcgen05.ld 32 columns at a time, scale, bias,
//               round, store.  Two accumulators let the epilogue of one tile
//               overlap the main loop of the next.
// Tile order: groups of row tiles (see pick_raster), so the tiles in flight
// form a square-ish block and share A and B panels in L2.
// Every wait is bounded (see mbar_wait); on a timeout the CTA drains its
// copies and MMAs, frees TMEM and exits, reporting through *status.
#include <cuda_bf16.h>
#include <stdlib.h>

#include "tc.cuh"

namespace fp8dl {

namespace g1 {
constexpr int BM = 128, BN = 256, BK = 128;  // BK in bytes = FP8 elements
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /* barriers */ + 1024 /* alignment slack */;
}  // namespace g1

struct GemmArgs {
    int64_t M, N, K;
    int raster_n;    // 1: groups of `group` column tiles, rows outer (B panels stay in L2)
    int64_t group;   // tiles per group along the grouped dimension
    int snake;       // 1: every other tile of a CTA pair reads its k-blocks last to first
    uint32_t idesc;
    const float *a_scale_inv, *b_scale_inv;
    const void *bias;
    int bias_dtype;  // -1 none, else fp8dl_hp_dtype
    void *D;
    int d_dtype;
    int32_t *status;
    // fused GELU + FP8 cast of the output (pair kernel, EPI = 1)
    uint8_t *q;            // [M x N] codes of g = GELU(D)
    uint8_t *q_t;          // [N x M] the same codes transposed (written by TMA from the CTA's staging)
    int q_fmt;             // fp8dl_fp8_dtype
    const float *q_scale;  // device float
    float *q_amax;         // device float, max-ed with max |g|, or NULL
    void *g_out;           // [M x N] bf16 g, or NULL
    // fused dGELU (EPI = 2): dh = dGELU(D, h) takes the place of g above
    const void *h_in;      // [M x N] bf16 h, the forward's GELU input
    float *ws;             // [ceil(M/32) x N] column sums of dh per 32-row group, or NULL
};

// Tile order.  Tiles come in groups of `group` tiles along one dimension; inside
// a group that dimension varies fastest.  The grouped dimension's operand
// panels stay resident in L2 while the other operand streams through once per
// group (pick_raster chooses the dimension and the group size).
__device__ __forceinline__ void tile_coords(int64_t tile, int64_t tiles_m, int64_t tiles_n, int raster_n,
                                            int64_t group, int64_t &tm, int64_t &tn) {
    const int64_t outer = raster_n ? tiles_m : tiles_n;  // tiles along the ungrouped dimension
    const int64_t inner = raster_n ? tiles_n : tiles_m;
    const int64_t per_group = group * outer;
    const int64_t g = tile / per_group;
    const int64_t first = g * group;
    const int64_t gsize = min(group, inner - first);
    const int64_t local = tile - g * per_group;
    const int64_t a = first + local % gsize, b = local / gsize;
    tm = raster_n ? b : a;
    tn = raster_n ? a : b;
}

__device__ __forceinline__ float load_bias(const void *bias, int dtype, int64_t n) {
    if (dtype == FP8DL_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(bias)[n]);
    return static_cast<const float *>(bias)[n];
}

__global__ void __launch_bounds__(g1::THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const GemmArgs args) {
    using namespace g1;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t *bar_area = smem + STAGES * STAGE_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(bar_area);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_m = (args.M + BM - 1) / BM, tiles_n = (args.N + BN - 1) / BN;
    const int64_t tiles = tiles_m * tiles_n;
    const int num_kb = (int)((args.K + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 4);
        }
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmap_a);
        tma_prefetch_map(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();  // set-up done; the previous kernel of the stream has completed
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                int64_t tm, tn;
                tile_coords(tile, tiles_m, tiles_n, args.raster_n, args.group, tm, tn);
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_expect_tx(fb, STAGE_BYTES);
                    uint8_t *sa = smem + s * STAGE_BYTES;
                    tma_load_2d(smem_u32(sa), &tmap_a, fb, kb * BK, (int32_t)(tm * BM));
                    tma_load_2d(smem_u32(sa + A_BYTES), &tmap_b, fb, kb * BK, (int32_t)(tn * BN));
                    issued++;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) {  // let every issued copy land before the CTA can exit
                for (int64_t i = issued - 1; i >= 0 && i >= issued - STAGES; i--)
                    mbar_drain(smem_u32(&full[i % STAGES]), (uint32_t)((i / STAGES) & 1));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true, any = false;
            uint32_t last_bar = 0, last_par = 0;
            const SDesc desc0 = sdesc_k_sw128_split(smem_u32(smem));  // stage 0's A tile
            for (int64_t tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                if (!mbar_wait(smem_u32(&tempty[acc]), aph ^ 1, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t lo_a = desc0.lo + (uint32_t)s * (STAGE_BYTES >> 4);
                    const uint32_t lo_b = lo_a + (A_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; kk++)  // K = 32 bytes per MMA: 2 descriptor units
                        umma_f8f6f4(d_tmem, sdesc_join(lo_a + 2 * kk, desc0.hi), sdesc_join(lo_b + 2 * kk, desc0.hi),
                                    args.idesc, (kb | kk) != 0);
                    umma_commit(smem_u32(&empty[s]));
                    any = true;
                    last_bar = smem_u32(&empty[s]);
                    last_par = ph;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&tfull[acc]));
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            if (!ok && any) mbar_drain(last_bar, last_par);  // MMAs in flight finish before TMEM is freed
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const float s = __fmul_rn(__ldg(args.a_scale_inv), __ldg(args.b_scale_inv));
        int acc = 0;
        uint32_t aph = 0;
        for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
            int64_t tm, tn;
            tile_coords(tile, tiles_m, tiles_n, args.raster_n, args.group, tm, tn);
            if (!mbar_wait(smem_u32(&tfull[acc]), aph, abort_flag, args.status)) break;
            tc_fence_after();
            const int64_t row = tm * BM + 32 * q + lane;
            const bool row_ok = row < args.M;
#pragma unroll 1
            for (int c = 0; c < BN / 32; c++) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (uint32_t)(acc * BN + c * 32) + ((uint32_t)(32 * q) << 16), r);
                tmem_ld_wait();
                const int64_t n0 = tn * BN + c * 32;
                if (row_ok && n0 < args.N) {
                    float v[32];
                    if (args.bias_dtype >= 0) {  // acc * s + bias with one rounding, as in the pair kernel
#pragma unroll
                        for (int j = 0; j < 32; j++)
                            v[j] = __fmaf_rn(__uint_as_float(r[j]), s,
                                             n0 + j < args.N ? load_bias(args.bias, args.bias_dtype, n0 + j) : 0.0f);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j++) v[j] = __fmul_rn(__uint_as_float(r[j]), s);
                    }
                    if (args.d_dtype == FP8DL_BF16) {
                        __nv_bfloat16 *drow = static_cast<__nv_bfloat16 *>(args.D) + row * args.N + n0;
#pragma unroll
                        for (int g = 0; g < 4; g++) {
                            if (n0 + 8 * g < args.N) {
                                uint32_t w[4];
#pragma unroll
                                for (int p = 0; p < 4; p++) {
                                    __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * g + 2 * p], v[8 * g + 2 * p + 1]);
                                    w[p] = *reinterpret_cast<uint32_t *>(&h);
                                }
                                *reinterpret_cast<uint4 *>(drow + 8 * g) = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    } else {
                        float *drow = static_cast<float *>(args.D) + row * args.N + n0;
#pragma unroll
                        for (int g = 0; g < 8; g++)
                            if (n0 + 4 * g < args.N)
                                *reinterpret_cast<float4 *>(drow + 4 * g) =
                                    make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
            if (++acc == 2) {
                acc = 0;
                aph ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}


// ---------------------------------------------------------------------------
// 2-SM variant: a cluster of two CTAs (one per SM) computes a 256x256 tile with
// tcgen05.mma.cta_group::2 (M=256, N=256, K=32).  Each CTA TMA-loads only its
// own halves — 128 rows of A and 128 rows of B (its half of N) — so every SM
// moves 32 KB per stage instead of 48 KB, and the shared-memory traffic per
// tensor cycle drops accordingly.  No data is multicast.
//   - Both CTAs' loads complete on the even ("leader") CTA's full barrier.
//   - The leader's single MMA thread issues for the pair; its commits arrive on
//     the empty/accumulator barriers at the same offset in both CTAs.
//   - Each CTA's epilogue drains its own 128 accumulator rows and releases
//     the accumulator on the leader's barrier (a remote arrive from the peer).
// ---------------------------------------------------------------------------
namespace g2 {
constexpr int BM = 128, BN = 256, BNH = 128, BK = 128;  // per-CTA rows of A and of B
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK, B_BYTES = BNH * BK, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
// epilogue warps: 4 (one per TMEM lane quarter) for the plain epilogue; 8 for the
// fused activation + cast ones, two per SM sub-partition, each draining 4 of the 8
// 32-column chunks of its lane quarter.  The MMA-issuing thread shares a sub-partition
// with them, and every epilogue instruction issued there delays it: with 16 warps
// (enough to hide all of the epilogue's latency) the tensor pipe lost more cycles than
// the shorter epilogue saved (measured: 8 warps take 3-4 % fewer cycles per launch).
__host__ __device__ constexpr int epi_warps(int epi) { return epi ? 8 : 4; }
__host__ __device__ constexpr int threads(int epi) { return 64 + 32 * epi_warps(epi); }
constexpr int QT_BYTES = BN * BM;  // transposed FP8 codes of one CTA's 128 x 256 output (fused epilogue)
// The fused epilogues stage their transposed codes in one tile beside the full operand ring.
__host__ __device__ constexpr int stages(int) { return STAGES; }
__host__ __device__ constexpr int qt_bufs(int epi) { return epi ? 1 : 0; }
constexpr int smem_bytes(int epi, int tn = BN) {
    return stages(epi) * (A_BYTES + tn / 2 * BK) + 1024 + qt_bufs(epi) * QT_BYTES + 1024;
}
}  // namespace g2

// EPI = 0: D = round(acc * s + bias).  EPI = 1 (fc1 of the LayerNormMLP): also
// g = bf16(GELU(D)), codes q = enc(fl32(g * scale)) row-major and transposed
// (the transposed codes of the CTA's 128 x 256 output are staged in shared
// memory and written with one TMA tensor store), and amax |g| — the cast that
// delayed scaling lets run inside the GEMM, its scale being known in advance.
// EPI = 2 (fc2 dgrad): the same with dh = bf16(dD * GELU'(h)) from the
// forward's h, D = dD optional, plus per-32-row column sums of dh (the fc1
// bias gradient before its final reduction).
// Bias of 32 consecutive output columns starting at n0 (0 beyond N).
__device__ __forceinline__ void load_bias32(const void *bias, int dtype, int64_t n0, int64_t N, float (&b)[32]) {
    if (n0 + 32 <= N && dtype == FP8DL_BF16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(bias) + n0);
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint4 u = __ldg(p + k);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                b[8 * k + 2 * q] = bf16_lo(w[q]);
                b[8 * k + 2 * q + 1] = bf16_hi(w[q]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j++) b[j] = n0 + j < N ? load_bias(bias, dtype, n0 + j) : 0.0f;
    }
}

// One step of a reduce-scatter over the 32 lanes: lane l keeps the half of
// y[0 .. 2O) selected by bit O of l and adds the partner's (lane l ^ O) copy
// of that half, leaving the sums in y[0 .. O).
template <int O, int L>
__device__ __forceinline__ void reduce_scatter_step(float (&y)[L], int lane) {
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < O; i++) {
        const float send = up ? y[i] : y[i + O];
        const float keep = up ? y[i + O] : y[i];
        y[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
}

// TN: the tile's columns, 256, or 128 for the plain GEMM of a small problem (more tiles to
// spread over the CTA pairs).
template <int EPI, int QF, int TN>  // QF: FP8 format of the fused epilogue's codes
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(g2::threads(EPI), 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_qt, const GemmArgs args) {
    using namespace g2;
    static_assert(TN == BN || (TN == BN / 2 && EPI == 0), "128-column tiles for the plain GEMM only");
    constexpr int TNH = TN / 2;                    // B rows per CTA
    constexpr int SB = A_BYTES + TNH * BK;         // one operand stage of one CTA
    constexpr int NST = stages(EPI);  // operand stages
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t *bar_area = smem + NST * SB;
    uint64_t *full = reinterpret_cast<uint64_t *>(bar_area);
    uint64_t *empty = full + NST;
    uint64_t *tfull = empty + NST;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint8_t *qt_stage = bar_area + 1024;  // EPI >= 1: one [256 columns][128 rows] code tile

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int64_t tiles_m = (args.M + 2 * BM - 1) / (2 * BM), tiles_n = (args.N + TN - 1) / TN;
    const int64_t tiles = tiles_m * tiles_n;
    const int num_kb = (int)((args.K + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; s++) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 2 * epi_warps(EPI));  // the epilogue warps of both CTAs
        }
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmap_a);
        tma_prefetch_map(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();  // set-up done; the previous kernel of the stream has completed
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ producer (both CTAs)
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            bool rev = false;  // this tile's k-blocks last to first (alternates per tile when snake)
            for (int64_t tile = pair; tile < tiles && ok; tile += npairs, rev = args.snake && !rev) {
                int64_t tm, tn;
                tile_coords(tile, tiles_m, tiles_n, args.raster_n, args.group, tm, tn);
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full[s]);
                    const uint32_t fb = mapa_shared(fb_local, 0);
                    if (leader) mbar_expect_tx(fb_local, 2 * SB);
                    uint8_t *sa = smem + s * SB;
                    const int32_t kx = (rev ? num_kb - 1 - kb : kb) * BK;
                    tma_load_2d_pair(smem_u32(sa), &tmap_a, fb, kx, (int32_t)(tm * 2 * BM + rank * BM));
                    tma_load_2d_pair(smem_u32(sa + A_BYTES), &tmap_b, fb, kx, (int32_t)(tn * TN + rank * TNH));
                    issued++;
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok && leader) {
                for (int64_t i = issued - 1; i >= 0 && i >= issued - NST; i--)
                    mbar_drain(smem_u32(&full[i % NST]), (uint32_t)((i / NST) & 1));
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {  // ----------------------------------------- MMA issuer (leader only)
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true, any = false;
            uint32_t last_bar = 0, last_par = 0;
            const SDesc desc0 = sdesc_k_sw128_split(smem_u32(smem));  // stage 0's A tile
            for (int64_t tile = pair; tile < tiles && ok; tile += npairs) {
                if (!mbar_wait(smem_u32(&tempty[acc]), aph ^ 1, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TN);
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t lo_a = desc0.lo + (uint32_t)s * (SB >> 4);
                    const uint32_t lo_b = lo_a + (A_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; kk++)  // K = 32 bytes per MMA: 2 descriptor units
                        umma_f8f6f4_pair(d_tmem, sdesc_join(lo_a + 2 * kk, desc0.hi),
                                         sdesc_join(lo_b + 2 * kk, desc0.hi), args.idesc, (kb | kk) != 0);
                    umma_commit_pair(smem_u32(&empty[s]), 0x3);
                    any = true;
                    last_bar = smem_u32(&empty[s]);
                    last_par = ph;
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit_pair(smem_u32(&tfull[acc]), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            if (!ok && any) mbar_drain(last_bar, last_par);
        }
    } else {  // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;                              // TMEM lane quarter
        const int part = (warp - 2) >> 2;                    // column part of the quarter
        constexpr int CHUNKS = TN / 32 / (epi_warps(EPI) / 4);  // 32-column chunks per warp
        constexpr int NEPI = 32 * epi_warps(EPI);            // epilogue threads
        const float sc = __fmul_rn(__ldg(args.a_scale_inv), __ldg(args.b_scale_inv));
        const float qscale = EPI ? __ldg(args.q_scale) : 0.0f;
        // 32-byte row stores where every row segment is 32-byte aligned: D's 32-column chunks of
        // bf16 (N a multiple of 16) and q's 32-byte chunks (N a multiple of 32)
        const bool d_v8 = (reinterpret_cast<uintptr_t>(args.D) & 31) == 0;
        const bool q_v8 = EPI && (reinterpret_cast<uintptr_t>(args.q) & 31) == 0 && (args.N & 31) == 0;
        // Transposed staging of the fused epilogue: qt_stage holds the CTA's q^T block as 256
        // rows of 128 bytes (one per output column) in the TMA 128-byte swizzle (16-byte chunk
        // k of row R at chunk k ^ (R & 7)).  A 4x4 byte transpose across each lane quad leaves
        // lane l with column 2(l & 1) + ((l >> 1) & 1) of its 4-column word for the quad's
        // rows 32q + 4(l >> 2) .. +3: one 32-bit store per word.

        float gmax = 0.0f;
        const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty[0]), 0), mapa_shared(smem_u32(&tempty[1]), 0)};
        int acc = 0;
        uint32_t aph = 0;
        int jt = 0;  // tiles drained by this CTA
        for (int64_t tile = pair; tile < tiles; tile += npairs) {
            int64_t tm, tn;
            tile_coords(tile, tiles_m, tiles_n, args.raster_n, args.group, tm, tn);
            const int64_t row = tm * 2 * BM + rank * BM + 32 * q + lane;
            const bool row_ok = row < args.M;
            const __nv_bfloat16 *hrow =
                EPI == 2 ? static_cast<const __nv_bfloat16 *>(args.h_in) + row * args.N : nullptr;
            if (EPI == 2 && row_ok && tn * TN + part * CHUNKS * 32 < args.N)  // this thread's h: one 128-byte line
                prefetch_l2(hrow + tn * TN + part * CHUNKS * 32);
            if (!mbar_wait(smem_u32(&tfull[acc]), aph, abort_flag, args.status)) break;
            tc_fence_after();
            uint8_t *qt_buf = qt_stage;
            if (EPI && jt > 0) {
                // The previous tile's store has finished reading the staging tile before anyone
                // writes it again.  Every epilogue warp got past the wait above (an abort stops
                // them all at the same tile's wait), so all of them reach this barrier.
                if (threadIdx.x == 64) bulk_wait_read();
                named_barrier(2, NEPI);
            }
#pragma unroll 1
            for (int cc = 0; cc < CHUNKS; cc++) {
                const int c = part * CHUNKS + cc;  // chunk of 32 columns within the tile
                const int64_t n0 = tn * TN + c * 32;
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (uint32_t)(acc * TN + c * 32) + ((uint32_t)(32 * q) << 16), r);
                float v[32];
                if (args.bias_dtype >= 0) {
                    float b[32];
                    load_bias32(args.bias, args.bias_dtype, n0, args.N, b);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {  // acc * s + bias, one rounding, two columns per instruction
                        const float2 a = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                        const float2 y = __ffma2_rn(a, f2(sc), make_float2(b[j], b[j + 1]));
                        v[j] = y.x;
                        v[j + 1] = y.y;
                    }
                } else {
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float2 y = __fmul2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), f2(sc));
                        v[j] = y.x;
                        v[j + 1] = y.y;
                    }
                }
                uint32_t hw[16];  // the bf16 output as packed pairs (also the activation's input)
                if (EPI || args.d_dtype == FP8DL_BF16) {
#pragma unroll
                    for (int p = 0; p < 16; p++) {
                        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * p], v[2 * p + 1]);
                        hw[p] = *reinterpret_cast<uint32_t *>(&h);
                    }
                }
                if (row_ok && n0 < args.N && args.D) {
                    if (EPI || args.d_dtype == FP8DL_BF16) {
                        __nv_bfloat16 *drow = static_cast<__nv_bfloat16 *>(args.D) + row * args.N + n0;
                        if (d_v8 && n0 + 32 <= args.N) {  // two full 32-byte sectors
                            st_global_v8(drow, hw[0], hw[1], hw[2], hw[3], hw[4], hw[5], hw[6], hw[7]);
                            st_global_v8(drow + 16, hw[8], hw[9], hw[10], hw[11], hw[12], hw[13], hw[14], hw[15]);
                        } else {
#pragma unroll
                            for (int g = 0; g < 4; g++)
                                if (n0 + 8 * g < args.N)
                                    *reinterpret_cast<uint4 *>(drow + 8 * g) =
                                        make_uint4(hw[4 * g], hw[4 * g + 1], hw[4 * g + 2], hw[4 * g + 3]);
                        }
                    } else {
                        float *drow = static_cast<float *>(args.D) + row * args.N + n0;
#pragma unroll
                        for (int g = 0; g < 8; g++)
                            if (n0 + 4 * g < args.N)
                                *reinterpret_cast<float4 *>(drow + 4 * g) =
                                    make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                    }
                }
                if (EPI) {
                    // y = GELU(D) (EPI 1) or dGELU(D, h) (EPI 2) in bf16, its codes, amax and the
                    // transposed staging.  Columns beyond N hold exact zeros (zero-filled B rows,
                    // zero bias) and so do rows beyond M in EPI 2 (no bias, h = 0); rows beyond M
                    // are kept out of the EPI 1 amax below.
                    // Groups of 8 columns: y, its bf16 store, codes and transposed staging; the
                    // EPI 2 column sums start at once (first reduce-scatter step, below).
                    uint32_t code[8];
                    float ys[16];  // EPI 2: y of columns 0-15, then the pair sums (j, j + 16)
                    float cmax = 0.0f;
                    const bool row_store = row_ok && n0 < args.N;
                    // EPI 2: h of 8 columns per group, loaded one group ahead (0 outside the matrix)
                    auto load_h8 = [&](int g) -> uint4 {
                        return (EPI == 2 && row_ok && n0 + 8 * g < args.N)
                                   ? __ldg(reinterpret_cast<const uint4 *>(hrow + n0 + 8 * g))
                                   : make_uint4(0u, 0u, 0u, 0u);
                    };
                    uint4 hcur = load_h8(0);
#pragma unroll
                    for (int g = 0; g < 4; g++) {
                        const uint4 hnext = g < 3 ? load_h8(g + 1) : make_uint4(0u, 0u, 0u, 0u);
                        const uint32_t hv[4] = {hcur.x, hcur.y, hcur.z, hcur.w};
                        uint32_t gw[4];
                        float y8[8];
#pragma unroll
                        for (int p = 0; p < 4; p++) {
                            const uint32_t w = hw[4 * g + p];
                            const float2 x = make_float2(bf16_lo(w), bf16_hi(w));
                            const float2 y = EPI == 1 ? gelu2_f32(x)
                                                      : dgelu2_f32(x, make_float2(bf16_lo(hv[p]), bf16_hi(hv[p])));
                            __nv_bfloat162 y2 = __floats2bfloat162_rn(y.x, y.y);
                            gw[p] = *reinterpret_cast<uint32_t *>(&y2);
                            y8[2 * p] = bf16_lo(gw[p]);
                            y8[2 * p + 1] = bf16_hi(gw[p]);
                        }
#pragma unroll
                        for (int j = 0; j < 8; j++) cmax = fmaxf(cmax, fabsf(y8[j]));
#pragma unroll
                        for (int h2 = 0; h2 < 2; h2++) {
                            const float *y4 = y8 + 4 * h2;
                            const float2 s01 = __fmul2_rn(make_float2(y4[0], y4[1]), f2(qscale));
                            const float2 s23 = __fmul2_rn(make_float2(y4[2], y4[3]), f2(qscale));
                            code[2 * g + h2] = pack4<QF>(s01.x, s01.y, s23.x, s23.y);
                        }
                        if (args.g_out && row_store && n0 + 8 * g < args.N)
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(args.g_out) + row * args.N + n0 +
                                                       8 * g) = make_uint4(gw[0], gw[1], gw[2], gw[3]);
#pragma unroll
                        for (int h2 = 0; h2 < 2; h2++) {
                            // 4x4 byte transpose across the lane quad (rows), then one 32-bit store
                            const uint32_t w = code[2 * g + h2];
                            const uint32_t a1 =
                                __byte_perm(w, __shfl_xor_sync(0xffffffffu, w, 1), (lane & 1) ? 0x3726u : 0x5140u);
                            const uint32_t t =
                                __byte_perm(a1, __shfl_xor_sync(0xffffffffu, a1, 2), (lane & 2) ? 0x3276u : 0x5410u);
                            const int col = c * 32 + 8 * g + 4 * h2 + (((lane & 1) << 1) | ((lane >> 1) & 1));
                            const int rb = 32 * q + 4 * (lane >> 2);  // first of the word's 4 rows
                            *reinterpret_cast<uint32_t *>(qt_buf + col * BM + (((rb >> 4) ^ (col & 7)) << 4) + (rb & 15)) = t;
                        }
                        if (EPI == 2) {
                            const bool up = (lane & 16) != 0;
#pragma unroll
                            for (int j = 0; j < 8; j++) {
                                if (g < 2) {
                                    ys[8 * g + j] = y8[j];
                                } else {  // column i + 16 meets column i: lane keeps one, trades the other
                                    const int i = 8 * (g - 2) + j;
                                    const float send = up ? ys[i] : y8[j];
                                    const float keep = up ? y8[j] : ys[i];
                                    ys[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                                }
                            }
                        }
                        hcur = hnext;
                    }
                    if (row_ok) gmax = fmaxf(gmax, cmax);
                    if (row_store) {
                        uint8_t *qrow = args.q + row * args.N + n0;
                        if (q_v8 && n0 + 32 <= args.N) {  // one full 32-byte sector
                            st_global_v8(qrow, code[0], code[1], code[2], code[3], code[4], code[5], code[6], code[7]);
                        } else {
                            if (n0 + 16 <= args.N)
                                *reinterpret_cast<uint4 *>(qrow) = make_uint4(code[0], code[1], code[2], code[3]);
                            if (n0 + 32 <= args.N)
                                *reinterpret_cast<uint4 *>(qrow + 16) = make_uint4(code[4], code[5], code[6], code[7]);
                        }
                    }
                    if (EPI == 2 && args.ws) {
                        // the rest of the reduce-scatter: lane l ends with column n0 + l summed
                        // over the warp's 32 rows
                        reduce_scatter_step<8>(ys, lane);
                        reduce_scatter_step<4>(ys, lane);
                        reduce_scatter_step<2>(ys, lane);
                        reduce_scatter_step<1>(ys, lane);
                        const int64_t row32 = tm * (2 * BM / 32) + rank * (BM / 32) + q;  // 32-row group
                        if (row32 * 32 < args.M && n0 + lane < args.N) args.ws[row32 * args.N + n0 + lane] = ys[0];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(smem_u32(&tempty[acc]));
                else
                    mbar_arrive_cluster(tempty_leader[acc]);
            }
            if (EPI) {  // the CTA's transposed codes: one TMA store of [256 columns x 128 rows]
                fence_proxy_async_smem();
                named_barrier(1, NEPI);
                if (threadIdx.x == 64 && tm * 2 * BM + rank * BM < args.M) {  // no store when all rows lie beyond M
                    tma_store_2d(&tmap_qt, smem_u32(qt_buf), (int32_t)(tm * 2 * BM + rank * BM), (int32_t)(tn * TN));
                    bulk_commit();
                }
            }
            jt++;
            if (++acc == 2) {
                acc = 0;
                aph ^= 1;
            }
        }
        if (EPI) {
            if (threadIdx.x == 64) bulk_wait_all();
            const float m = warp_max(gmax);
            if (lane == 0 && args.q_amax) atomic_max_nonneg(args.q_amax, m);
        }
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    __syncwarp();
    cluster_sync();  // the peer's shared memory and TMEM stay live until the pair is done
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: one thread waits, through mbar_wait, on a
// barrier phase that completes only if `arrive_first` is set.
// ---------------------------------------------------------------------------
__global__ void wait_selftest_kernel(long long budget, int arrive_first, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        mbar_fence_init();
        if (arrive_first) mbar_arrive(smem_u32(&bar));
        if (mbar_wait(smem_u32(&bar), 0, &abort_flag, status, budget)) atomicExch(reinterpret_cast<int *>(status), 0);
    }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

fp8dl_status encode_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                               uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                               CUtensorMapSwizzle swizzle) {
    if (!g_encode_tiled) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return fail(FP8DL_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP8DL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FP8DL_OK;
}

// Tile order: groups of `group` tiles along one dimension, that dimension fastest inside a
// group.  The tiles in flight step through K together, so what one wave reads from DRAM
// grows with the number of distinct A and B panels it spans; a square-ish block of
// concurrent tiles (group ~ sqrt of the tiles in flight, counted in elements) keeps that
// smallest.  Each group reads the other dimension's operand once more.  With square tiles
// (the pair kernel's 256 x 256) the groups run along the dimension with fewer tiles: fewer
// groups, fewer re-reads.  Measured at 16384 x 4096 x 16384: row groups 0.564 ms, column
// groups 0.554 ms; the reverse at 4096 x 16384 x 16384.  Their group size follows the panel
// size (256 x K bytes): with K <= 8192 groups of 16 re-read less and still fit the wave's
// panels in L2 (16384 x 16384 x 4096: 0.560 ms with 8, 0.546 with 16, 0.591 with 64; the
// fused GELU/dGELU epilogues 1-1.4 % faster with 16); with K = 16384 groups of 8 are
// fastest (6: +1.3 %, 12: +0.9 %).  The 128 x 256 tiles keep row groups of 16.  An order that keeps a
// whole operand "resident" instead streamed the other operand's panels through L2 and
// raised DRAM reads (16384x16384x4096: 601 MB -> 927 MB).  FP8DL_GEMM_RASTER=m|n and
// FP8DL_GEMM_GROUP=g override the order (testing).
void pick_raster(int64_t M, int64_t N, int64_t K, int64_t tile_m, int64_t tile_n, int &raster_n, int64_t &group) {
    const int64_t tiles_m = (M + tile_m - 1) / tile_m, tiles_n = (N + tile_n - 1) / tile_n;
    raster_n = tile_m == tile_n && tiles_n < tiles_m ? 1 : 0;
    group = tile_m >= tile_n ? (K <= 8192 ? 16 : 8) : 16;  // pair tiles: 16 / 8 by K; 128x256 tiles: 16
    const char *r = getenv("FP8DL_GEMM_RASTER");
    const char *g = getenv("FP8DL_GEMM_GROUP");
    if (r && r[0] == 'n') raster_n = 1;
    if (r && r[0] == 'm') raster_n = 0;
    if (g && atoll(g) > 0) group = atoll(g);
}

// K order: a CTA (pair) that runs several tiles reads the k-blocks of every other tile
// last to first.  The tiles in flight step through K together and share panels with the
// next wave's tiles (the grouped dimension's panels); when the next tile starts where the
// last one ended, its first k-blocks are the ones most recently read, still in L2, instead
// of the oldest ones, which a wave's panels have pushed out.  Each tile's sum then runs
// over K in one of two orders, fixed by the tile's position in the CTA's sequence: the
// result is the same on every call with the same grid and tiling.  Used only when the
// launch has at least two waves (so short GEMMs keep one order whatever their tile width)
// and K > 8192.  Measured DRAM reads per launch: 16384 x 4096 x 16384 1001 -> 928 MB,
// MXFP8 16384 x 8192 x 28672 4085 -> 3509 MB; with K = 4096 or 8192, whose panels already
// stay in L2 across waves, they rose by 1-8 %.  FP8DL_GEMM_SNAKE=0 turns it off (testing).
int pick_snake(int64_t tiles, int64_t ctas, int64_t K) {
    const char *v = getenv("FP8DL_GEMM_SNAKE");
    if (v && v[0] == '0') return 0;
    return tiles >= 2 * ctas && K > 8192 ? 1 : 0;
}

static fp8dl_status check_gemm_common(int64_t M, int64_t N, int64_t K, int64_t mult, const void *A, const void *B,
                                      const void *bias, int32_t bias_dtype, const void *D, int32_t d_dtype,
                                      bool d_required = true) {
    FP8DL_CHECK_ARG(A && B && (D || !d_required), "A, B and D must be non-NULL");
    FP8DL_CHECK_ARG(d_dtype == FP8DL_BF16 || d_dtype == FP8DL_F32, "d_dtype must be FP8DL_BF16 or FP8DL_F32");
    FP8DL_CHECK_ARG(!bias || bias_dtype == FP8DL_BF16 || bias_dtype == FP8DL_F32,
                    "bias_dtype must be FP8DL_BF16 or FP8DL_F32");
    if (!dim_ok(M, mult) || !dim_ok(N, mult) || !dim_ok(K, mult))
        return fail(FP8DL_ERR_SHAPE, "M, N, K (%lld, %lld, %lld) must be positive multiples of %lld", (long long)M,
                    (long long)N, (long long)K, (long long)mult);
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(bias))
        return fail(FP8DL_ERR_ALIGN, "A, B, bias and D must be 16-byte aligned");
    return FP8DL_OK;
}

}  // namespace fp8dl

using namespace fp8dl;

extern "C" fp8dl_status fp8dl_wait_selftest(int64_t budget_cycles, int32_t arrive_first, int32_t *dev_status,
                                            fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8dl_wait_selftest");
    FP8DL_CHECK_ARG(dev_status != nullptr, "dev_status is NULL");
    FP8DL_CHECK_ARG(budget_cycles >= 0 && budget_cycles <= (int64_t(1) << 32), "budget_cycles must be in [0, 2^32]");
    if (!aligned16(dev_status)) return fail(FP8DL_ERR_ALIGN, "dev_status must be 16-byte aligned");
    FP8DL_TRY(current_device(nullptr, nullptr));
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((long long)budget_cycles, arrive_first ? 1 : 0,
                                                             dev_status);
    note_launch();
    return check_launch("fp8dl_wait_selftest");
}

namespace fp8dl {

// Per-device launch state of the GEMM kernels.  g_pair_clusters is written before the
// release store of g_attr_set; callers read it after gemm_device_setup returned.
static std::atomic<bool> g_attr_set[64];
static int g_pair_clusters[64];

static fp8dl_status gemm_device_setup(int dev, int sms) {
    if (g_attr_set[dev].load(std::memory_order_acquire)) return FP8DL_OK;
    std::lock_guard<std::mutex> lock(init_mutex());
    if (g_attr_set[dev].load(std::memory_order_relaxed)) return FP8DL_OK;
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, g1::SMEM_BYTES);
    const void *pair_kernels[] = {(const void *)fp8_gemm_pair_kernel<0, 0, g2::BN>,
                                  (const void *)fp8_gemm_pair_kernel<1, FP8DL_E4M3, g2::BN>,
                                  (const void *)fp8_gemm_pair_kernel<1, FP8DL_E5M2, g2::BN>,
                                  (const void *)fp8_gemm_pair_kernel<2, FP8DL_E4M3, g2::BN>,
                                  (const void *)fp8_gemm_pair_kernel<2, FP8DL_E5M2, g2::BN>,
                                  (const void *)fp8_gemm_pair_kernel<0, 0, g2::BN / 2>};
    const int pair_epi[] = {0, 1, 1, 2, 2, 0}, pair_tn[] = {g2::BN, g2::BN, g2::BN, g2::BN, g2::BN, g2::BN / 2};
    for (int k = 0; k < 6 && e == cudaSuccess; k++)
        e = cudaFuncSetAttribute(pair_kernels[k], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g2::smem_bytes(pair_epi[k], pair_tn[k]));
    if (e != cudaSuccess) return fail(FP8DL_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    // how many CTA pairs can be resident at once (both pair kernels hold one CTA per SM)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms / 2 * 2), 1, 1);
    cfg.blockDim = dim3(g2::threads(1), 1, 1);
    cfg.dynamicSmemBytes = g2::smem_bytes(1);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, (const void *)fp8_gemm_pair_kernel<1, FP8DL_E4M3, g2::BN>, &cfg);
    if (e != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        clusters = 0;  // the pair kernels are not used on this device
    }
    g_pair_clusters[dev] = clusters;
    g_attr_set[dev].store(true, std::memory_order_release);
    return FP8DL_OK;
}

// The 2-SM pair kernel runs when the problem has two 128-row halves per tile and
// pairs can be resident; FP8DL_GEMM_VARIANT=1sm|2sm overrides (testing).
static bool gemm_use_pair(int dev, int64_t M) {
    const char *v = getenv("FP8DL_GEMM_VARIANT");
    const int forced = (v && v[0] == '1') ? 1 : (v && v[0] == '2') ? 2 : 0;
    return g_pair_clusters[dev] > 0 && (forced == 2 || (forced == 0 && M > g1::BM));
}

// Shared launch path of fp8_gemm (epi = 0), fp8_gemm_gelu_cast (epi = 1) and
// fp8_gemm_dgelu_cast (epi = 2); the fused epilogues exist in the pair kernel only.
static fp8dl_status launch_gemm(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype, int64_t M,
                                int64_t N, int64_t K, GemmArgs &args, int epi, int dev, int sms, bool use_pair,
                                cudaStream_t stream) {
    CUtensorMap ta, tb, tq;
    const bool pdl = short_call_flops(2.0 * (double)M * (double)N * (double)K);
    // Instruction descriptor, kind::f8f6f4: D fp32 (bit 4), A type bits 7-9, B type bits 10-12
    // (0 = E4M3, 1 = E5M2), both K-major, N>>3 at bits 17-22, M>>4 at bits 24-28
    // (M = 128 for one CTA, 256 for a CTA pair; N = the tile's columns).
    const uint32_t idesc_ab = (1u << 4) | ((uint32_t)a_dtype << 7) | ((uint32_t)b_dtype << 10);
    const uint32_t idesc_base = idesc_ab | ((uint32_t)(g1::BN >> 3) << 17);
    FP8DL_TRY(encode_tmap_2d_u8(&ta, A, (uint64_t)K, (uint64_t)M, (uint64_t)K, g1::BK, g1::BM,
                                CU_TENSOR_MAP_SWIZZLE_128B));
    if (use_pair) {
        // Tile columns: 256, or 128 for a short plain GEMM (under 64 GFLOP) whose 256-column
        // tiles would not fill two waves of the resident pairs: twice the tiles to spread.  For
        // a long GEMM with few tiles the narrow tiles lose more than they gain (twice the MMA
        // issues and A loads per FLOP: a 2048-token Llama micro-batch step ran 21 % slower).
        // FP8DL_GEMM_TILE_N=256|128 overrides (testing).
        const int64_t tiles256 = ((M + 2 * g2::BM - 1) / (2 * g2::BM)) * ((N + g2::BN - 1) / g2::BN);
        int tn = (epi == 0 && pdl && tiles256 < 2 * (int64_t)g_pair_clusters[dev]) ? g2::BN / 2 : g2::BN;
        const char *tv = getenv("FP8DL_GEMM_TILE_N");
        if (epi == 0 && tv && atoi(tv) == 128) tn = g2::BN / 2;
        if (tv && atoi(tv) == 256) tn = g2::BN;
        // A in 128-row boxes and B in tn/2-row boxes: each CTA of a pair loads its own halves
        FP8DL_TRY(encode_tmap_2d_u8(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)K, g2::BK, (uint32_t)(tn / 2),
                                    CU_TENSOR_MAP_SWIZZLE_128B));
        if (epi) {
            // q^T [N x M] codes, stored in boxes of 128 rows of the output (inner) x 256 columns
            FP8DL_TRY(encode_tmap_2d_u8(&tq, args.q_t, (uint64_t)M, (uint64_t)N, (uint64_t)M, g2::BM, g2::BN,
                                        CU_TENSOR_MAP_SWIZZLE_128B));
        } else {
            tq = ta;  // unused
        }
        args.idesc = idesc_ab | ((uint32_t)(tn >> 3) << 17) | ((uint32_t)(2 * g2::BM >> 4) << 24);
        pick_raster(M, N, K, 2 * g2::BM, tn, args.raster_n, args.group);
        const int64_t tiles = ((M + 2 * g2::BM - 1) / (2 * g2::BM)) * ((N + tn - 1) / tn);
        const int64_t pairs = tiles < g_pair_clusters[dev] ? tiles : g_pair_clusters[dev];
        const unsigned grid = (unsigned)(2 * pairs);
        args.snake = tn == g2::BN ? pick_snake(tiles, pairs, K) : 0;
        const bool e4 = args.q_fmt == FP8DL_E4M3;
        if (epi == 2 && e4)
            (void)launch_kernel(fp8_gemm_pair_kernel<2, FP8DL_E4M3, g2::BN>, grid, g2::threads(2), g2::smem_bytes(2), stream, 0, pdl, ta, tb, tq, args);
        else if (epi == 2)
            (void)launch_kernel(fp8_gemm_pair_kernel<2, FP8DL_E5M2, g2::BN>, grid, g2::threads(2), g2::smem_bytes(2), stream, 0, pdl, ta, tb, tq, args);
        else if (epi == 1 && e4)
            (void)launch_kernel(fp8_gemm_pair_kernel<1, FP8DL_E4M3, g2::BN>, grid, g2::threads(1), g2::smem_bytes(1), stream, 0, pdl, ta, tb, tq, args);
        else if (epi == 1)
            (void)launch_kernel(fp8_gemm_pair_kernel<1, FP8DL_E5M2, g2::BN>, grid, g2::threads(1), g2::smem_bytes(1), stream, 0, pdl, ta, tb, tq, args);
        else if (tn == g2::BN)
            (void)launch_kernel(fp8_gemm_pair_kernel<0, 0, g2::BN>, grid, g2::threads(0), g2::smem_bytes(0), stream, 0, pdl, ta, tb, tq, args);
        else
            (void)launch_kernel(fp8_gemm_pair_kernel<0, 0, g2::BN / 2>, grid, g2::threads(0),
                                g2::smem_bytes(0, g2::BN / 2), stream, 0, pdl, ta, tb, tq, args);
        note_launch();
        return check_launch(epi == 2 ? "fp8_gemm_dgelu_cast(pair)"
                                     : epi == 1 ? "fp8_gemm_gelu_cast(pair)" : "fp8_gemm(pair)");
    }
    FP8DL_TRY(encode_tmap_2d_u8(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)K, g1::BK, g1::BN,
                                CU_TENSOR_MAP_SWIZZLE_128B));
    args.idesc = idesc_base | ((uint32_t)(g1::BM >> 4) << 24);
    pick_raster(M, N, K, g1::BM, g1::BN, args.raster_n, args.group);
    args.snake = 0;  // the one-CTA kernel reads K first to last
    const int64_t tiles = ((M + g1::BM - 1) / g1::BM) * ((N + g1::BN - 1) / g1::BN);
    const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
    (void)launch_kernel(fp8_gemm_kernel, grid, g1::THREADS, g1::SMEM_BYTES, stream, 0, pdl, ta, tb, args);
    note_launch();
    return check_launch("fp8_gemm");
}

static fp8dl_status gemm_args(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype, int64_t M,
                              int64_t N, int64_t K, const float *a_scale_inv, const float *b_scale_inv,
                              const void *bias, int32_t bias_dtype, void *D, int32_t d_dtype, int32_t *dev_status,
                              GemmArgs &args, bool d_required = true) {
    FP8DL_TRY(check_gemm_common(M, N, K, 16, A, B, bias, bias_dtype, D, d_dtype, d_required));
    FP8DL_CHECK_ARG((a_dtype == FP8DL_E4M3 || a_dtype == FP8DL_E5M2) && (b_dtype == FP8DL_E4M3 || b_dtype == FP8DL_E5M2),
                    "a_dtype and b_dtype must be E4M3 or E5M2");
    FP8DL_CHECK_ARG(a_scale_inv && b_scale_inv, "a_scale_inv and b_scale_inv must be non-NULL");
    args = GemmArgs{};
    args.M = M;
    args.N = N;
    args.K = K;
    args.a_scale_inv = a_scale_inv;
    args.b_scale_inv = b_scale_inv;
    args.bias = bias;
    args.bias_dtype = bias ? bias_dtype : -1;
    args.D = D;
    args.d_dtype = d_dtype;
    args.status = dev_status;
    return FP8DL_OK;
}

}  // namespace fp8dl

extern "C" fp8dl_status fp8_gemm(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype, int64_t M,
                                 int64_t N, int64_t K, const float *a_scale_inv, const float *b_scale_inv,
                                 const void *bias, int32_t bias_dtype, void *D, int32_t d_dtype, int32_t *dev_status,
                                 fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_gemm");
    GemmArgs args;
    FP8DL_TRY(gemm_args(A, a_dtype, B, b_dtype, M, N, K, a_scale_inv, b_scale_inv, bias, bias_dtype, D, d_dtype,
                        dev_status, args));
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    FP8DL_TRY(gemm_device_setup(dev, sms));
    return launch_gemm(A, a_dtype, B, b_dtype, M, N, K, args, 0, dev, sms, gemm_use_pair(dev, M), (cudaStream_t)stream);
}

extern "C" fp8dl_status fp8_gemm_gelu_cast(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype,
                                           int64_t M, int64_t N, int64_t K, const float *a_scale_inv,
                                           const float *b_scale_inv, const void *bias, int32_t bias_dtype, void *H,
                                           int32_t q_dtype, const float *q_scale, uint8_t *q, uint8_t *q_t,
                                           float *q_amax, void *g, int32_t *dev_status, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_gemm_gelu_cast");
    GemmArgs args;
    FP8DL_TRY(gemm_args(A, a_dtype, B, b_dtype, M, N, K, a_scale_inv, b_scale_inv, bias, bias_dtype, H, FP8DL_BF16,
                        dev_status, args));
    FP8DL_CHECK_ARG(q_dtype == FP8DL_E4M3 || q_dtype == FP8DL_E5M2, "q_dtype must be E4M3 or E5M2");
    FP8DL_CHECK_ARG(q && q_t && q_scale, "q, q_t and q_scale must be non-NULL");
    if (!aligned16(q) || !aligned16(q_t) || !aligned16(g))
        return fail(FP8DL_ERR_ALIGN, "q, q_t and g must be 16-byte aligned");
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    FP8DL_TRY(gemm_device_setup(dev, sms));
    if (!gemm_use_pair(dev, M)) {
        // one-CTA kernel: the GEMM, then the GELU + cast kernel over its output
        FP8DL_TRY(launch_gemm(A, a_dtype, B, b_dtype, M, N, K, args, 0, dev, sms, false, (cudaStream_t)stream));
        return fp8_gelu_cast(H, M, N, q_dtype, q_scale, q, q_t, q_amax, g, stream);
    }
    args.q = q;
    args.q_t = q_t;
    args.q_fmt = q_dtype;
    args.q_scale = q_scale;
    args.q_amax = q_amax;
    args.g_out = g;
    return launch_gemm(A, a_dtype, B, b_dtype, M, N, K, args, 1, dev, sms, true, (cudaStream_t)stream);
}

extern "C" size_t fp8_gemm_dgelu_workspace_size(int64_t M, int64_t N) {
    if (M <= 0 || N <= 0) return 0;
    return (size_t)((M + 31) / 32) * (size_t)N * sizeof(float);
}

extern "C" fp8dl_status fp8_gemm_dgelu_cast(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype,
                                            int64_t M, int64_t N, int64_t K, const float *a_scale_inv,
                                            const float *b_scale_inv, const void *h, void *dg, int32_t q_dtype,
                                            const float *q_scale, uint8_t *q, uint8_t *q_t, float *q_amax,
                                            float *dbias, void *workspace, size_t workspace_bytes, void *dh,
                                            int32_t *dev_status, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_gemm_dgelu_cast");
    GemmArgs args;
    FP8DL_TRY(gemm_args(A, a_dtype, B, b_dtype, M, N, K, a_scale_inv, b_scale_inv, nullptr, FP8DL_BF16, dg, FP8DL_BF16,
                        dev_status, args, /*d_required=*/false));
    FP8DL_CHECK_ARG(q_dtype == FP8DL_E4M3 || q_dtype == FP8DL_E5M2, "q_dtype must be E4M3 or E5M2");
    FP8DL_CHECK_ARG(h && q && q_t && q_scale, "h, q, q_t and q_scale must be non-NULL");
    if (!aligned16(h) || !aligned16(q) || !aligned16(q_t) || !aligned16(dh))
        return fail(FP8DL_ERR_ALIGN, "h, q, q_t and dh must be 16-byte aligned");
    if (dbias) {
        if (!workspace || workspace_bytes < fp8_gemm_dgelu_workspace_size(M, N))
            return fail(FP8DL_ERR_WORKSPACE, "dbias needs a workspace of %zu bytes (got %zu)",
                        fp8_gemm_dgelu_workspace_size(M, N), workspace ? workspace_bytes : (size_t)0);
        if (!aligned16(workspace)) return fail(FP8DL_ERR_ALIGN, "workspace must be 16-byte aligned");
    }
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    FP8DL_TRY(gemm_device_setup(dev, sms));
    if (g_pair_clusters[dev] < 1)
        return fail(FP8DL_ERR_UNSUPPORTED_DEVICE, "fp8_gemm_dgelu_cast needs resident CTA-pair clusters");
    args.q = q;
    args.q_t = q_t;
    args.q_fmt = q_dtype;
    args.q_scale = q_scale;
    args.q_amax = q_amax;
    args.g_out = dh;
    args.h_in = h;
    args.ws = dbias ? static_cast<float *>(workspace) : nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    FP8DL_TRY(launch_gemm(A, a_dtype, B, b_dtype, M, N, K, args, 2, dev, sms, true, st));
    if (dbias) {
        colsum_reduce(args.ws, (M + 31) / 32, N, dbias, st, short_call_flops(2.0 * (double)M * (double)N * (double)K));
        FP8DL_TRY(check_launch("fp8_gemm_dgelu_cast(dbias reduce)"));
    }
    return FP8DL_OK;
}
