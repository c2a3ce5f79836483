// mxfp8.cu — MXFP8 (block-scaled FP8): quantisation and the block-scaled GEMM.
//
// MXFP8 is named by the Transformer Engine README ("亮点": MXFP8 and NVFP4 on
// Blackwell) without a definition.  Reading used throughout this library:
// E4M3 data, one E8M0 scale (a biased power of two, byte = e + 127) per 32
// consecutive elements along the reduction axis.  The block exponent is the
// power-of-two form of the per-tensor scale FP8_MAX/amax of
// "FP8 低精度训练：Transformer Engine 简析" §三.1: the smallest e with
// amax_b * 2^-e <= 448, so a block's largest element never saturates.
#include <cuda_bf16.h>

#include "tc.cuh"

namespace fp8dl {

// ---------------------------------------------------------------------------
// quantisation
// ---------------------------------------------------------------------------
// Smallest e with amax * 2^-e <= 448 (= 1.75 * 2^8), clamped to [-127, 127];
// amax = 0 gives 0.  Computed exactly from the bits: amax = (1 + m/2^23) * 2^E,
// and 1 + m/2^23 <= 1.75 exactly when m <= 0x600000.
__device__ __forceinline__ int e8m0_exponent(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    if (bits == 0u) return 0;
    int E;
    uint32_t m;
    const uint32_t ef = bits >> 23;
    if (ef == 0u) {  // subnormal: bits * 2^-149
        const int p = 31 - __clz(bits);
        E = p - 149;
        m = (bits << (23 - p)) & 0x7FFFFFu;
    } else {
        E = (int)ef - 127;
        m = bits & 0x7FFFFFu;
    }
    int e = (m <= 0x600000u) ? E - 8 : E - 7;
    return max(-127, min(127, e));
}

// 2^-e as an exact fp32 (2^-127 is subnormal).
__device__ __forceinline__ float pow2_neg(int e) {
    return e <= 126 ? __int_as_float((127 - e) << 23) : __int_as_float(0x00400000);
}

// Byte offset of scale S[r][b] in the tiled scale layout (128-row x 4-block
// tiles of 512 bytes; kg = number of 4-block groups per row = ceil(NB / 4)).
// Inside a tile, row r sits in 16-byte line r % 32 at word (r % 128) / 32, and
// block b at byte b % 4 of that word: the order tcgen05.cp .32x128b.warpx4
// moves into tensor memory for the block-scaled MMA.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t b, int64_t kg) {
    return ((r >> 7) * kg + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3);
}

constexpr int MQ_ROWS = 32, MQ_COLS = 256, MQ_THREADS = 256;

// Shared-memory staging of a 32 x 256 tile, rows of 256*ESZ bytes.  16-byte
// chunks are XOR-swizzled by their 32-element block index so that the row pass
// (8 threads reading 8 different blocks of one row) and the column pass (32
// threads reading one row's consecutive elements) are both conflict free.
template <int ESZ>
__device__ __forceinline__ int mq_chunk(int cc) {
    constexpr int PER_BLOCK = 32 * ESZ / 16;
    return cc ^ ((cc / PER_BLOCK) & 7);
}

template <int XKIND>
__device__ __forceinline__ float mq_load(const uint8_t *tile, int r, int c) {
    constexpr int ESZ = XKIND == FP8DL_BF16 ? 2 : 4;
    const int byte = c * ESZ;
    const uint8_t *p = tile + r * MQ_COLS * ESZ + mq_chunk<ESZ>(byte >> 4) * 16 + (byte & 15);
    if (XKIND == FP8DL_BF16) return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(p)) << 16);
    return *reinterpret_cast<const float *>(p);
}

// 32 consecutive elements of row r starting at block b, as fp32.
template <int XKIND>
__device__ __forceinline__ void mq_load_block(const uint8_t *tile, int r, int b, float (&v)[32]) {
    constexpr int ESZ = XKIND == FP8DL_BF16 ? 2 : 4;
    constexpr int PER_BLOCK = 32 * ESZ / 16;
#pragma unroll
    for (int j = 0; j < PER_BLOCK; j++) {
        const uint4 u = *reinterpret_cast<const uint4 *>(tile + r * MQ_COLS * ESZ +
                                                         mq_chunk<ESZ>(b * PER_BLOCK + j) * 16);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (XKIND == FP8DL_BF16) {
                v[8 * j + 2 * q] = bf16_lo(w[q]);
                v[8 * j + 2 * q + 1] = bf16_hi(w[q]);
            } else {
                v[4 * j + q] = __uint_as_float(w[q]);
            }
        }
    }
}

// One tile = 32 rows x 256 cols.  Phase 1 stages the tile in shared memory
// with coalesced 16-byte loads; the row pass gives each thread one 1x32
// block, the column pass one 32x1 block (one column of the tile).
template <int XKIND>
__global__ void __launch_bounds__(MQ_THREADS) mxfp8_quantize_kernel(const void *__restrict__ x, int64_t rows,
                                                                    int64_t cols, uint8_t *__restrict__ row_q,
                                                                    uint8_t *__restrict__ row_s,
                                                                    uint8_t *__restrict__ col_q,
                                                                    uint8_t *__restrict__ col_s) {
    constexpr int ESZ = XKIND == FP8DL_BF16 ? 2 : 4;
    constexpr int CHUNKS_PER_ROW = MQ_COLS * ESZ / 16;
    constexpr int CHUNKS = MQ_ROWS * CHUNKS_PER_ROW;
    __shared__ __align__(16) uint8_t tile[MQ_ROWS * MQ_COLS * ESZ];
    const int t = threadIdx.x;
    const int64_t tiles_c = (cols + MQ_COLS - 1) / MQ_COLS;
    const int64_t tiles = (rows / MQ_ROWS) * tiles_c;
    for (int64_t tl = blockIdx.x; tl < tiles; tl += gridDim.x) {
        const int64_t r0 = (tl / tiles_c) * MQ_ROWS, c0 = (tl % tiles_c) * MQ_COLS;
        const int valid_cols = (int)min((int64_t)MQ_COLS, cols - c0);
        for (int k = t; k < CHUNKS; k += MQ_THREADS) {
            const int r = k / CHUNKS_PER_ROW, cc = k % CHUNKS_PER_ROW;
            if (cc * 16 / ESZ < valid_cols) {
                const uint8_t *src = static_cast<const uint8_t *>(x) + ((r0 + r) * cols + c0) * ESZ + cc * 16;
                *reinterpret_cast<uint4 *>(tile + (r * MQ_COLS) * ESZ + mq_chunk<ESZ>(cc) * 16) = ldg_stream(src);
            }
        }
        __syncthreads();
        if (row_q) {  // row pass: thread -> (row r, block b)
            const int r = t >> 3, b = t & 7;
            if (32 * b < valid_cols) {
                float v[32];
                float amax = 0.0f;
                mq_load_block<XKIND>(tile, r, b, v);
#pragma unroll
                for (int j = 0; j < 32; j++) amax = fmaxf(amax, fabsf(v[j]));
                const int e = e8m0_exponent(amax);
                const float mult = pow2_neg(e);
                uint32_t w[8];
#pragma unroll
                for (int q = 0; q < 8; q++)
                    w[q] = pack4<FP8DL_E4M3>(__fmul_rn(v[4 * q], mult), __fmul_rn(v[4 * q + 1], mult),
                                             __fmul_rn(v[4 * q + 2], mult), __fmul_rn(v[4 * q + 3], mult));
                uint8_t *dst = row_q + (r0 + r) * cols + c0 + 32 * b;
                reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                row_s[sf_offset(r0 + r, c0 / 32 + b, (cols / 32 + 3) / 4)] = (uint8_t)(e + 127);
            }
        }
        if (col_q) {  // column pass: thread -> column t of the tile
            if (t < valid_cols) {
                float v[32];
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    v[j] = mq_load<XKIND>(tile, j, t);
                    amax = fmaxf(amax, fabsf(v[j]));
                }
                const int e = e8m0_exponent(amax);
                const float mult = pow2_neg(e);
                uint32_t w[8];
#pragma unroll
                for (int q = 0; q < 8; q++)
                    w[q] = pack4<FP8DL_E4M3>(__fmul_rn(v[4 * q], mult), __fmul_rn(v[4 * q + 1], mult),
                                             __fmul_rn(v[4 * q + 2], mult), __fmul_rn(v[4 * q + 3], mult));
                uint8_t *dst = col_q + (c0 + t) * rows + r0;
                reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                col_s[sf_offset(c0 + t, r0 / 32, (rows / 32 + 3) / 4)] = (uint8_t)(e + 127);
            }
        }
        __syncthreads();
    }
}

// Scale entries outside the matrix (rows R..Rp-1, or blocks NB..NBp-1 of a
// real row) are set to 127 (2^0): the GEMM then multiplies the zero-filled
// padding data by 1.
__global__ void sf_pad_kernel(uint8_t *__restrict__ s, int64_t R, int64_t NB, int64_t Rp, int64_t NBp) {
    const int64_t n1 = (Rp - R) * NBp, n2 = R * (NBp - NB);
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    int64_t r, b;
    if (i < n1) {
        r = R + i / NBp;
        b = i % NBp;
    } else if (i < n1 + n2) {
        i -= n1;
        r = i / (NBp - NB);
        b = NB + i % (NBp - NB);
    } else {
        return;
    }
    s[sf_offset(r, b, NBp / 4)] = 127;
}

static void launch_sf_pad(uint8_t *s, int64_t R, int64_t NB, cudaStream_t st) {
    const int64_t Rp = (R + 127) / 128 * 128, NBp = (NB + 3) / 4 * 4;
    const int64_t n = (Rp - R) * NBp + R * (NBp - NB);
    if (n > 0) sf_pad_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(s, R, NB, Rp, NBp);
}


// ---------------------------------------------------------------------------
// Block-scaled GEMM: tcgen05.mma kind::mxf8f6f4 with E8M0 scales in TMEM.
//
//   warp 0      producer: TMA of the 128x128 A and 256x128 B data tiles and
//               bulk copies of their tiled scales (512 B for A, 2 x 512 B for
//               B) into a 4-stage ring.
//   warp 1      TMEM owner and MMA issuer: per stage, tcgen05.cp moves the
//               scales into tensor memory (32x128b, replicated to the four
//               lane quarters), then 4 MMAs of K=32 select scale byte kk of
//               each row with the scale-factor ids of the instruction
//               descriptor.
//   warps 2-9   epilogue: one 128x256 fp32 accumulator; each warp drains 128
//               columns of its lane quarter into registers (packed bf16),
//               releases the accumulator for the next tile, then stores.
// TMEM: columns 0-255 accumulator, 256 + 16*s: scales of stage s
// (4 columns for A, 8 for B).
// ---------------------------------------------------------------------------
namespace mx {
constexpr int BM = 128, BN = 256, BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK, AB_BYTES = A_BYTES + B_BYTES;
constexpr int SFA_BYTES = 512, SFB_BYTES = 1024, SF_BYTES = SFA_BYTES + SFB_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 256, SF_COLS_PER_STAGE = 16;
constexpr int GROUP_M = 16;
constexpr int SMEM_BYTES = STAGES * AB_BYTES + STAGES * SF_BYTES + 1024 /* barriers */ + 1024 /* alignment */;
}  // namespace mx

struct MxArgs {
    int64_t M, N, K;
    const uint8_t *sfa, *sfb;
    int64_t kg;       // 4-block groups per row of the scale layout = ceil(K / 128)
    int64_t sfb_rows; // 128-row scale tiles of B = ceil(N / 128)
    uint32_t idesc;   // without the scale-factor ids
    const void *bias;
    int bias_dtype;
    void *D;
    int d_dtype;
    int32_t *status;
};

__device__ __forceinline__ void mx_tile_coords(int64_t tile, int64_t tiles_m, int64_t tiles_n, int64_t &tm,
                                               int64_t &tn) {
    const int64_t per_group = (int64_t)mx::GROUP_M * tiles_n;
    const int64_t g = tile / per_group;
    const int64_t first_m = g * mx::GROUP_M;
    const int64_t gsize = min((int64_t)mx::GROUP_M, tiles_m - first_m);
    const int64_t local = tile - g * per_group;
    tm = first_m + local % gsize;
    tn = local / gsize;
}

__device__ __forceinline__ float mx_bias(const void *bias, int dtype, int64_t n) {
    if (dtype == FP8DL_BF16) return __uint_as_float((uint32_t)static_cast<const uint16_t *>(bias)[n] << 16);
    return static_cast<const float *>(bias)[n];
}

__global__ void __launch_bounds__(mx::THREADS, 1)
    mxfp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      const MxArgs args) {
    using namespace mx;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t *sf_area = smem + STAGES * AB_BYTES;
    uint8_t *bar_area = sf_area + STAGES * SF_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(bar_area);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 1);
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
        mbar_init(smem_u32(tfull), 1);
        mbar_init(smem_u32(tempty), EPI_WARPS);
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

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ producer
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                int64_t tm, tn;
                mx_tile_coords(tile, tiles_m, tiles_n, tm, tn);
                const bool sfb1 = 2 * tn + 1 < args.sfb_rows;
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_expect_tx(fb, AB_BYTES + SFA_BYTES + (sfb1 ? 1024 : 512));
                    uint8_t *sa = smem + s * AB_BYTES;
                    uint8_t *sf = sf_area + s * SF_BYTES;
                    tma_load_2d(smem_u32(sa), &tmap_a, fb, kb * BK, (int32_t)(tm * BM));
                    tma_load_2d(smem_u32(sa + A_BYTES), &tmap_b, fb, kb * BK, (int32_t)(tn * BN));
                    bulk_load(smem_u32(sf), args.sfa + (tm * args.kg + kb) * 512, 512, fb);
                    bulk_load(smem_u32(sf + 512), args.sfb + ((2 * tn) * args.kg + kb) * 512, 512, fb);
                    if (sfb1) bulk_load(smem_u32(sf + 1024), args.sfb + ((2 * tn + 1) * args.kg + kb) * 512, 512, fb);
                    issued++;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) {
                for (int64_t i = issued - 1; i >= 0 && i >= issued - STAGES; i--)
                    mbar_drain(smem_u32(&full[i % STAGES]), (uint32_t)((i / STAGES) & 1));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ------------------------------------------------ MMA issuer
            int s = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true, any = false;
            uint32_t last_bar = 0, last_par = 0;
            for (int64_t tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                if (!mbar_wait(smem_u32(tempty), aph ^ 1, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * AB_BYTES), sb = sa + A_BYTES;
                    const uint32_t sf = smem_u32(sf_area + s * SF_BYTES);
                    const uint32_t t_sfa = tmem_base + (uint32_t)(SF_COL0 + s * SF_COLS_PER_STAGE);
                    const uint32_t t_sfb = t_sfa + 4;
                    tmem_cp_32x128b_warpx4(t_sfa, sdesc_rows16(sf));
                    tmem_cp_32x128b_warpx4(t_sfb, sdesc_rows16(sf + 512));
                    tmem_cp_32x128b_warpx4(t_sfb + 4, sdesc_rows16(sf + 1024));
#pragma unroll
                    for (int kk = 0; kk < BK / 32; kk++) {
                        // scale-factor ids: byte kk of each scale word, for A (bits 29-30) and B (bits 4-5)
                        const uint32_t idesc = args.idesc | ((uint32_t)kk << 29) | ((uint32_t)kk << 4);
                        umma_mxf8f6f4(tmem_base, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32), idesc,
                                      t_sfa, t_sfb, (kb | kk) != 0);
                    }
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
                umma_commit(smem_u32(tfull));
                aph ^= 1;
            }
            if (!ok && any) mbar_drain(last_bar, last_par);
        }
    } else {  // ------------------------------------------------------------ epilogue
        const int q = warp & 3, h = (warp - 2) >> 2;  // lane quarter, column half
        uint32_t aph = 0;
        for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
            int64_t tm, tn;
            mx_tile_coords(tile, tiles_m, tiles_n, tm, tn);
            if (!mbar_wait(smem_u32(tfull), aph, abort_flag, args.status)) break;
            tc_fence_after();
            const int64_t row = tm * BM + 32 * q + lane;
            const int64_t n_base = tn * BN + 128 * h;
            const uint32_t taddr = tmem_base + (uint32_t)(128 * h) + ((uint32_t)(32 * q) << 16);
            if (args.d_dtype == FP8DL_BF16) {
                uint32_t packed[64];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + 32 * c, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        float lo = __uint_as_float(r[2 * j]), hi = __uint_as_float(r[2 * j + 1]);
                        const int64_t n = n_base + 32 * c + 2 * j;
                        if (args.bias_dtype >= 0) {
                            if (n < args.N) lo += mx_bias(args.bias, args.bias_dtype, n);
                            if (n + 1 < args.N) hi += mx_bias(args.bias, args.bias_dtype, n + 1);
                        }
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                        packed[16 * c + j] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(tempty));
                if (row < args.M) {
                    __nv_bfloat16 *drow = static_cast<__nv_bfloat16 *>(args.D) + row * args.N;
#pragma unroll
                    for (int g = 0; g < 16; g++) {
                        const int64_t n = n_base + 8 * g;
                        if (n < args.N)
                            *reinterpret_cast<uint4 *>(drow + n) =
                                make_uint4(packed[4 * g], packed[4 * g + 1], packed[4 * g + 2], packed[4 * g + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 4; c++) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + 32 * c, r);
                    tmem_ld_wait();
                    if (row < args.M) {
                        float *drow = static_cast<float *>(args.D) + row * args.N;
#pragma unroll
                        for (int g = 0; g < 8; g++) {
                            const int64_t n = n_base + 32 * c + 4 * g;
                            if (n < args.N) {
                                float v[4];
#pragma unroll
                                for (int j = 0; j < 4; j++) {
                                    v[j] = __uint_as_float(r[4 * g + j]);
                                    if (args.bias_dtype >= 0) v[j] += mx_bias(args.bias, args.bias_dtype, n + j);
                                }
                                *reinterpret_cast<float4 *>(drow + n) = make_float4(v[0], v[1], v[2], v[3]);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(tempty));
            }
            aph ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace fp8dl

using namespace fp8dl;

extern "C" {

size_t mxfp8_scale_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)((rows + 127) / 128) * (size_t)((cols / 32 + 3) / 4) * 512;
}

fp8dl_status mxfp8_quantize(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, uint8_t *row_q,
                            uint8_t *row_s, uint8_t *col_q, uint8_t *col_s, fp8dl_stream_t stream) {
    FP8DL_CHECK_ARG(x != nullptr, "x is NULL");
    FP8DL_CHECK_ARG(x_dtype == FP8DL_F32 || x_dtype == FP8DL_BF16, "x_dtype must be FP8DL_F32 or FP8DL_BF16");
    FP8DL_CHECK_ARG((row_q == nullptr) == (row_s == nullptr), "row_q and row_s must both be given or both NULL");
    FP8DL_CHECK_ARG((col_q == nullptr) == (col_s == nullptr), "col_q and col_s must both be given or both NULL");
    FP8DL_CHECK_ARG(row_q || col_q, "nothing to compute: all outputs are NULL");
    if (!dim_ok(rows, 32) || !dim_ok(cols, 32))
        return fail(FP8DL_ERR_SHAPE, "rows (%lld) and cols (%lld) must be positive multiples of 32",
                    (long long)rows, (long long)cols);
    if (!aligned16(x) || !aligned16(row_q) || !aligned16(col_q))
        return fail(FP8DL_ERR_ALIGN, "x, row_q and col_q must be 16-byte aligned");
    int sms = 0;
    FP8DL_TRY(current_device(nullptr, &sms));
    const int64_t tiles = (rows / MQ_ROWS) * ((cols + MQ_COLS - 1) / MQ_COLS);
    const int64_t max_ctas = (int64_t)sms * 8;
    const unsigned grid = (unsigned)(tiles < max_ctas ? tiles : max_ctas);
    if (x_dtype == FP8DL_BF16)
        mxfp8_quantize_kernel<FP8DL_BF16><<<grid, MQ_THREADS, 0, (cudaStream_t)stream>>>(x, rows, cols, row_q, row_s,
                                                                                          col_q, col_s);
    else
        mxfp8_quantize_kernel<FP8DL_F32><<<grid, MQ_THREADS, 0, (cudaStream_t)stream>>>(x, rows, cols, row_q, row_s,
                                                                                         col_q, col_s);
    FP8DL_TRY(check_launch("mxfp8_quantize"));
    if (row_s) launch_sf_pad(row_s, rows, cols / 32, (cudaStream_t)stream);
    if (col_s) launch_sf_pad(col_s, cols, rows / 32, (cudaStream_t)stream);
    return check_launch("mxfp8_quantize(scale padding)");
}

fp8dl_status mxfp8_gemm(const uint8_t *A, const uint8_t *A_s, const uint8_t *B, const uint8_t *B_s, int64_t M,
                        int64_t N, int64_t K, const void *bias, int32_t bias_dtype, void *D, int32_t d_dtype,
                        int32_t *dev_status, fp8dl_stream_t stream) {
    FP8DL_CHECK_ARG(A && A_s && B && B_s && D, "A, A_s, B, B_s and D must be non-NULL");
    FP8DL_CHECK_ARG(d_dtype == FP8DL_BF16 || d_dtype == FP8DL_F32, "d_dtype must be FP8DL_BF16 or FP8DL_F32");
    FP8DL_CHECK_ARG(!bias || bias_dtype == FP8DL_BF16 || bias_dtype == FP8DL_F32,
                    "bias_dtype must be FP8DL_BF16 or FP8DL_F32");
    if (!dim_ok(M, 32) || !dim_ok(N, 32) || !dim_ok(K, 32))
        return fail(FP8DL_ERR_SHAPE, "M, N, K (%lld, %lld, %lld) must be positive multiples of 32", (long long)M,
                    (long long)N, (long long)K);
    if (!aligned16(A) || !aligned16(B) || !aligned16(A_s) || !aligned16(B_s) || !aligned16(D) || !aligned16(bias))
        return fail(FP8DL_ERR_ALIGN, "A, A_s, B, B_s, bias and D must be 16-byte aligned");
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    CUtensorMap ta, tb;
    FP8DL_TRY(encode_tmap_2d_u8(&ta, A, (uint64_t)K, (uint64_t)M, (uint64_t)K, mx::BK, mx::BM,
                                CU_TENSOR_MAP_SWIZZLE_128B));
    FP8DL_TRY(encode_tmap_2d_u8(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)K, mx::BK, mx::BN,
                                CU_TENSOR_MAP_SWIZZLE_128B));
    MxArgs args;
    args.M = M;
    args.N = N;
    args.K = K;
    args.sfa = A_s;
    args.sfb = B_s;
    args.kg = (K / 32 + 3) / 4;
    args.sfb_rows = (N + 127) / 128;
    // Block-scaled instruction descriptor: A and B E4M3 (bits 7-9, 10-12 = 0), K-major,
    // N>>3 at bits 17-22, scale type E8M0 (bit 23), M>>4 at bits 24-28; the
    // scale-factor ids (bits 4-5 for B, 29-30 for A) are added per MMA.
    args.idesc = ((uint32_t)(mx::BN >> 3) << 17) | (1u << 23) | ((uint32_t)(mx::BM >> 4) << 24);
    args.bias = bias;
    args.bias_dtype = bias ? bias_dtype : -1;
    args.D = D;
    args.d_dtype = d_dtype;
    args.status = dev_status;
    static bool attr_set[64] = {};
    if (!attr_set[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(mxfp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mx::SMEM_BYTES);
        if (e != cudaSuccess) return fail(FP8DL_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        attr_set[dev] = true;
    }
    const int64_t tiles = ((M + mx::BM - 1) / mx::BM) * ((N + mx::BN - 1) / mx::BN);
    const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
    mxfp8_gemm_kernel<<<grid, mx::THREADS, mx::SMEM_BYTES, (cudaStream_t)stream>>>(ta, tb, args);
    return check_launch("mxfp8_gemm");
}

}  // extern "C"
