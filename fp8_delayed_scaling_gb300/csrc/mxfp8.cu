// mxfp8.cu — MXFP8 (block-scaled FP8): quantisation and the block-scaled GEMM.
//
// MXFP8 is named by the Transformer Engine README ("亮点": MXFP8 and NVFP4 on
// Blackwell) without a definition.  Reading used throughout this library:
// E4M3 data, one E8M0 scale (a biased power of two, byte = e + 127) per 32
// consecutive elements along the reduction axis.  The block exponent is the
// power-of-two form of the per-tensor scale FP8_MAX/amax of
// "FP8 低精度训练：Transformer Engine 简析" §三.1: the smallest e with
// amax_b * 2^-e <= 448, so a block's largest element never saturates.
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
                row_s[(r0 + r) * (cols / 32) + (c0 / 32) + b] = (uint8_t)(e + 127);
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
                col_s[(c0 + t) * (rows / 32) + r0 / 32] = (uint8_t)(e + 127);
            }
        }
        __syncthreads();
    }
}

}  // namespace fp8dl

using namespace fp8dl;

extern "C" {

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
    return check_launch("mxfp8_quantize");
}

fp8dl_status mxfp8_gemm(const uint8_t *A, const uint8_t *A_s, const uint8_t *B, const uint8_t *B_s, int64_t M,
                        int64_t N, int64_t K, const void *bias, int32_t bias_dtype, void *D, int32_t d_dtype,
                        int32_t *dev_status, fp8dl_stream_t stream) {
    (void)A; (void)A_s; (void)B; (void)B_s; (void)M; (void)N; (void)K; (void)bias; (void)bias_dtype; (void)D;
    (void)d_dtype; (void)dev_status; (void)stream;
    return fail(FP8DL_ERR_INVALID_ARG, "mxfp8_gemm: not built yet");
}

}  // extern "C"
