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

void pick_raster(int64_t M, int64_t N, int64_t K, int64_t tile_m, int64_t tile_n, int &raster_n, int64_t &group);
int pick_snake(int64_t tiles, int64_t ctas, int64_t K);

// ---------------------------------------------------------------------------
// quantisation
// ---------------------------------------------------------------------------
// Smallest e with amax * 2^-e <= 448 (= 1.75 * 2^8), clamped to [-127, 127];
// amax = 0 gives 0.  From the bits: a normal amax = (1 + m/2^23) * 2^(E-127)
// with 1 + m/2^23 <= 1.75 exactly when m <= 0x600000, so e = E - 135 + (m >
// 0x600000).  Every subnormal amax (E = 0) gives e <= -134, i.e. -127 after
// the clamp, and the largest amax (E = 255) gives e <= 121, so only the lower
// clamp is ever active.
__device__ __forceinline__ int e8m0_exponent(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    int e = (int)(bits >> 23) - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    e = max(e, -127);
    return bits == 0u ? 0 : e;
}

// 2^-e as an exact fp32 for e in [-127, 121] (the exponents e8m0_exponent gives).
__device__ __forceinline__ float pow2_neg(int e) { return __int_as_float((127 - e) << 23); }

// Byte offset of scale S[r][b] in the tiled scale layout (128-row x 4-block
// tiles of 512 bytes; kg = number of 4-block groups per row = ceil(NB / 4)).
// Inside a tile, row r sits in 16-byte line r % 32 at word (r % 128) / 32, and
// block b at byte b % 4 of that word: the order tcgen05.cp .32x128b.warpx4
// moves into tensor memory for the block-scaled MMA.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t b, int64_t kg) {
    return ((r >> 7) * kg + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3);
}

// ---------------------------------------------------------------------------
// Quantisation kernel.  A CTA tile is 128 x 128 elements; the CTA streams its
// tiles through a three-stage shared-memory ring filled with cp.async by all
// threads, so the next two tiles are in flight while one is converted.
// Each warp converts a 32-row x 64-column part of the tile (two 32 x 32
// blocks side by side).  From shared memory each lane
// takes 8 rows x 8 columns: lane bits 0-1 = 8-column chunk, bits 2-3 = 8-row
// chunk, bit 4 = which 32 x 32 block.  Row-block amaxes reduce over lane bits
// 0-1, column-block amaxes over bits 2-3 (shuffles within each block's 16
// lanes).  Row-wise codes leave as 8-byte row pieces, column-wise codes after
// an in-register 8 x 8 byte transpose as 8-byte pieces of the transposed rows
// (four lanes fill each 32-byte sector).
// ---------------------------------------------------------------------------
constexpr int MQ_THREADS = 256, MQ_STAGES = 3;

// Transpose a 4x4 byte block held as 4 row words: word c of the result holds
// column c, rows in byte order.
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&o)[4]) {
    const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(c, d, 0x5140);
    const uint32_t t2 = __byte_perm(a, b, 0x7362), t3 = __byte_perm(c, d, 0x7362);
    o[0] = __byte_perm(t0, t1, 0x5410);
    o[1] = __byte_perm(t0, t1, 0x7632);
    o[2] = __byte_perm(t2, t3, 0x5410);
    o[3] = __byte_perm(t2, t3, 0x7632);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stage one CTA tile (128 rows x 128 columns) into shared memory with 16-byte
// cp.async chunks; rows and columns past the matrix are skipped.
template <int ESZ>
__device__ __forceinline__ void mq_stage(uint8_t *buf, const void *x, int64_t rows, int64_t cols, int64_t r0,
                                         int64_t c0) {
    constexpr int ROW_BYTES = 128 * ESZ, PER_ROW = ROW_BYTES / 16, CHUNKS = 128 * PER_ROW;
    const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(buf);
#pragma unroll
    for (int k = 0; k < CHUNKS / MQ_THREADS; k++) {
        const int ch = threadIdx.x + MQ_THREADS * k, r = ch / PER_ROW, c = ch % PER_ROW;
        if (r0 + r < rows && c0 + c * 16 / ESZ < cols)
            cp_async16(sbuf + r * ROW_BYTES + c * 16,
                       static_cast<const char *>(x) + ((r0 + r) * cols + c0) * ESZ + c * 16);
    }
}

// ws (optional): column sums of x per 128-row tile, ws[tile row][column] (the bias
// gradient before its final reduction over tile rows).  Per tile: each lane sums its 8
// rows, the four lanes of a 32-row band add theirs (two shuffles), and the four bands of
// the tile are added in band order, so the sums are the same on every run.
template <int XKIND, bool DBIAS>
__global__ void __launch_bounds__(MQ_THREADS) mxfp8_quantize_kernel(const void *__restrict__ x, int64_t rows,
                                                                    int64_t cols, uint8_t *__restrict__ row_q,
                                                                    uint8_t *__restrict__ row_s,
                                                                    uint8_t *__restrict__ col_q,
                                                                    uint8_t *__restrict__ col_s,
                                                                    float *__restrict__ ws) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    constexpr int ESZ = XKIND == FP8DL_BF16 ? 2 : 4;
    constexpr int ROW_BYTES = 128 * ESZ, STAGE = 128 * ROW_BYTES;
    extern __shared__ __align__(16) uint8_t mq_smem[];
    // Scales of one CTA tile: exactly one 512-byte tile of the tiled scale layout per
    // orientation (128 rows x 4 blocks).  Double-buffered; written out one iteration later.
    __shared__ __align__(16) uint8_t sf_tile[2][2][512];  // [buffer][row-wise, column-wise]
    __shared__ __align__(16) float band_sum[DBIAS ? 2 : 1][4][128];  // [buffer][32-row band][column] (DBIAS)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cc = lane & 3, rr = (lane >> 2) & 3, sub = lane >> 4;
    const int wr = warp >> 1, wc = warp & 1;  // this warp's 32-row band and 64-column half of the tile
    const int64_t tiles_c = (cols + 127) / 128, tiles = ((rows + 127) / 128) * tiles_c;
    const int64_t kg_row = (cols / 32 + 3) / 4, kg_col = (rows / 32 + 3) / 4;
    // in-tile position of this lane's 8 x 8 piece
    const int prow = 32 * wr + 8 * rr, pcol = 64 * wc + 32 * sub + 8 * cc;
    // byte of the in-tile scale layout for (row r, block b) of a 128-row x 4-block tile
    auto sf_byte = [](int r, int b) { return (r & 31) * 16 + (r >> 5) * 4 + b; };
    for (int k = threadIdx.x; k < 2 * 2 * 512 / 4; k += MQ_THREADS) reinterpret_cast<uint32_t *>(sf_tile)[k] = 0x7F7F7F7Fu;
#pragma unroll
    for (int k = 0; k < MQ_STAGES - 1; k++) {
        const int64_t t0 = blockIdx.x + (int64_t)k * gridDim.x;
        if (t0 < tiles) mq_stage<ESZ>(mq_smem + k * STAGE, x, rows, cols, (t0 / tiles_c) * 128, (t0 % tiles_c) * 128);
        cp_async_commit();
    }
    int stage = 0, sfb = 0;
    int64_t prev_tile = -1;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t nt = tile + (int64_t)(MQ_STAGES - 1) * gridDim.x;
        const int ns = stage == 0 ? MQ_STAGES - 1 : stage - 1;  // the stage consumed one iteration ago
        if (nt < tiles) mq_stage<ESZ>(mq_smem + ns * STAGE, x, rows, cols, (nt / tiles_c) * 128, (nt % tiles_c) * 128);
        cp_async_commit();
        cp_async_wait<MQ_STAGES - 1>();
        __syncthreads();  // the current stage is complete for every thread; the previous tile's scales are final
        if (prev_tile >= 0 && threadIdx.x < 64) {  // write the previous tile's two scale tiles, 16 bytes per thread
            const int o = threadIdx.x & 31, which = threadIdx.x >> 5;
            const int64_t ptr = prev_tile / tiles_c, ptc = prev_tile % tiles_c;
            uint8_t *dst = which == 0 ? row_s + (ptr * kg_row + ptc) * 512 : col_s + (ptc * kg_col + ptr) * 512;
            uint4 *src = reinterpret_cast<uint4 *>(sf_tile[sfb ^ 1][which]) + o;
            if ((which == 0 ? row_q : col_q) != nullptr) *(reinterpret_cast<uint4 *>(dst) + o) = *src;
            *src = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);  // padding default for reuse
        }
        if constexpr (DBIAS) {
            if (prev_tile >= 0 && threadIdx.x >= 128) {  // the previous tile's column sums, bands in order
                const int c = threadIdx.x - 128;
                const int64_t ptr = prev_tile / tiles_c, pc = (prev_tile % tiles_c) * 128 + c;
                const float(*bs)[128] = band_sum[sfb ^ 1];
                if (pc < cols) ws[ptr * cols + pc] = ((bs[0][c] + bs[1][c]) + bs[2][c]) + bs[3][c];
            }
        }
        const int64_t tr0 = (tile / tiles_c) * 128, tc0 = (tile % tiles_c) * 128;
        const bool ok = tr0 + 32 * wr < rows && tc0 + 64 * wc + 32 * sub < cols;  // whole 32 x 32 block present
        const uint8_t *sb = mq_smem + stage * STAGE + prow * ROW_BYTES + pcol * ESZ;
        float2 v[8][4];     // v[i][q]: columns 2q, 2q+1 of row i of the lane's piece
        uint32_t wq[8][4];  // bf16 input: the same pairs as bf16x2 words
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint8_t *p = sb + i * ROW_BYTES;
            if (ESZ == 2) {
                const uint4 u = *reinterpret_cast<const uint4 *>(p);
                wq[i][0] = u.x, wq[i][1] = u.y, wq[i][2] = u.z, wq[i][3] = u.w;
#pragma unroll
                for (int q = 0; q < 4; q++) v[i][q] = make_float2(bf16_lo(wq[i][q]), bf16_hi(wq[i][q]));
            } else {
                const uint4 u0 = *reinterpret_cast<const uint4 *>(p), u1 = *reinterpret_cast<const uint4 *>(p + 16);
                v[i][0] = make_float2(__uint_as_float(u0.x), __uint_as_float(u0.y));
                v[i][1] = make_float2(__uint_as_float(u0.z), __uint_as_float(u0.w));
                v[i][2] = make_float2(__uint_as_float(u1.x), __uint_as_float(u1.y));
                v[i][3] = make_float2(__uint_as_float(u1.z), __uint_as_float(u1.w));
            }
        }
        __syncthreads();  // the stage may be refilled once every thread has read it
        if constexpr (DBIAS) {
            // bands of the tile beyond the matrix (rows are a multiple of 32) add zeros
            const bool band_ok = tr0 + 32 * wr < rows;
            float cs[8];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float2 a = v[0][q];
#pragma unroll
                for (int i = 1; i < 8; i++) a = __fadd2_rn(a, v[i][q]);
                cs[2 * q] = band_ok ? a.x : 0.0f;
                cs[2 * q + 1] = band_ok ? a.y : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 8; j++) {
                cs[j] += __shfl_xor_sync(0xffffffffu, cs[j], 4);
                cs[j] += __shfl_xor_sync(0xffffffffu, cs[j], 8);
            }
            if (rr == 0) {
                float4 *dst = reinterpret_cast<float4 *>(&band_sum[sfb][wr][pcol]);
                dst[0] = make_float4(cs[0], cs[1], cs[2], cs[3]);
                dst[1] = make_float4(cs[4], cs[5], cs[6], cs[7]);
            }
        }
        float rmax[8], cmax[8];
        if constexpr (ESZ == 2) {  // |x| maxima on the bf16x2 words, two columns per instruction
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t r2 = bf16x2_absmax(bf16x2_absmax(wq[i][0], wq[i][1]), bf16x2_absmax(wq[i][2], wq[i][3]));
                rmax[i] = fmaxf(fabsf(bf16_lo(r2)), fabsf(bf16_hi(r2)));
            }
#pragma unroll
            for (int q = 0; q < 4; q++) {
                uint32_t c2 = wq[0][q];
#pragma unroll
                for (int i = 1; i < 8; i++) c2 = bf16x2_absmax(c2, wq[i][q]);
                cmax[2 * q] = fabsf(bf16_lo(c2));
                cmax[2 * q + 1] = fabsf(bf16_hi(c2));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                rmax[i] = 0.0f;
                cmax[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float a = fabsf(v[i][q].x), b = fabsf(v[i][q].y);
                    rmax[i] = fmaxf(rmax[i], fmaxf(a, b));
                    cmax[2 * q] = fmaxf(cmax[2 * q], a);
                    cmax[2 * q + 1] = fmaxf(cmax[2 * q + 1], b);
                }
        }
#pragma unroll
        for (int i = 0; i < 8; i++) {
            rmax[i] = fmaxf(rmax[i], __shfl_xor_sync(0xffffffffu, rmax[i], 1));
            rmax[i] = fmaxf(rmax[i], __shfl_xor_sync(0xffffffffu, rmax[i], 2));
            cmax[i] = fmaxf(cmax[i], __shfl_xor_sync(0xffffffffu, cmax[i], 4));
            cmax[i] = fmaxf(cmax[i], __shfl_xor_sync(0xffffffffu, cmax[i], 8));
        }
        if (ok && row_q) {
            uint8_t *qrow = row_q + (tr0 + prow) * cols + tc0 + pcol;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int e = e8m0_exponent(rmax[i]);
                const float2 m = f2(pow2_neg(e));
                const float2 a = __fmul2_rn(v[i][0], m), b = __fmul2_rn(v[i][1], m);
                const float2 c = __fmul2_rn(v[i][2], m), d = __fmul2_rn(v[i][3], m);
                const uint32_t lo = pack4<FP8DL_E4M3>(a.x, a.y, b.x, b.y);
                const uint32_t hi = pack4<FP8DL_E4M3>(c.x, c.y, d.x, d.y);
                *reinterpret_cast<uint2 *>(qrow + i * cols) = make_uint2(lo, hi);
                if (cc == 0) sf_tile[sfb][0][sf_byte(prow + i, pcol >> 5)] = (uint8_t)(e + 127);
            }
        }
        if (ok && col_q) {
            float m[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int e = e8m0_exponent(cmax[j]);
                m[j] = pow2_neg(e);
                if (rr == 0) sf_tile[sfb][1][sf_byte(pcol + j, prow >> 5)] = (uint8_t)(e + 127);
            }
            uint8_t *qcol = col_q + (tc0 + pcol) * rows + tr0 + prow;
#pragma unroll
            for (int half = 0; half < 2; half++) {  // columns 4*half .. 4*half+3
                uint32_t wcode[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const float2 a = __fmul2_rn(v[i][2 * half], make_float2(m[4 * half], m[4 * half + 1]));
                    const float2 b = __fmul2_rn(v[i][2 * half + 1], make_float2(m[4 * half + 2], m[4 * half + 3]));
                    wcode[i] = pack4<FP8DL_E4M3>(a.x, a.y, b.x, b.y);
                }
                uint32_t lo[4], hi[4];
                transpose4x4(wcode[0], wcode[1], wcode[2], wcode[3], lo);
                transpose4x4(wcode[4], wcode[5], wcode[6], wcode[7], hi);
#pragma unroll
                for (int j = 0; j < 4; j++)
                    *reinterpret_cast<uint2 *>(qcol + (4 * half + j) * rows) = make_uint2(lo[j], hi[j]);
            }
        }
        stage = stage == MQ_STAGES - 1 ? 0 : stage + 1;
        prev_tile = tile;
        sfb ^= 1;
    }
    cp_async_wait<0>();
    __syncthreads();
    if constexpr (DBIAS) {
        if (prev_tile >= 0 && threadIdx.x >= 128) {  // the last tile's column sums
            const int c = threadIdx.x - 128;
            const int64_t ptr = prev_tile / tiles_c, pc = (prev_tile % tiles_c) * 128 + c;
            const float(*bs)[128] = band_sum[sfb ^ 1];
            if (pc < cols) ws[ptr * cols + pc] = ((bs[0][c] + bs[1][c]) + bs[2][c]) + bs[3][c];
        }
    }
    if (prev_tile >= 0 && threadIdx.x < 64) {  // the last tile's scales
        const int o = threadIdx.x & 31, which = threadIdx.x >> 5;
        const int64_t ptr = prev_tile / tiles_c, ptc = prev_tile % tiles_c;
        uint8_t *dst = which == 0 ? row_s + (ptr * kg_row + ptc) * 512 : col_s + (ptc * kg_col + ptr) * 512;
        if ((which == 0 ? row_q : col_q) != nullptr)
            *(reinterpret_cast<uint4 *>(dst) + o) = *(reinterpret_cast<const uint4 *>(sf_tile[sfb ^ 1][which]) + o);
    }
}

// Scale entries outside the matrix (rows R..Rp-1, or blocks NB..NBp-1 of a
// real row) are set to 127 (2^0): the GEMM then multiplies the zero-filled
// padding data by 1.
__global__ void sf_pad_kernel(uint8_t *__restrict__ s, int64_t R, int64_t NB, int64_t Rp, int64_t NBp) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
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

static void launch_sf_pad(uint8_t *s, int64_t R, int64_t NB, cudaStream_t st, bool pdl) {
    const int64_t Rp = (R + 127) / 128 * 128, NBp = (NB + 3) / 4 * 4;
    const int64_t n = (Rp - R) * NBp + R * (NBp - NB);
    if (n > 0) {
        (void)launch_kernel(sf_pad_kernel, (unsigned)((n + 255) / 256), 256, 0, st, 0, pdl, s, R, NB, Rp, NBp);
        note_launch();
    }
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
constexpr int SMEM_BYTES = STAGES * AB_BYTES + STAGES * SF_BYTES + 1024 /* barriers */ + 1024 /* alignment */;
}  // namespace mx

struct MxArgs {
    int64_t M, N, K;
    int raster_n;
    int64_t group;
    int snake;        // 1: every other tile of a CTA reads its k-blocks last to first
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

__device__ __forceinline__ void mx_tile_coords(int64_t tile, int64_t tiles_m, int64_t tiles_n, int raster_n,
                                               int64_t group, int64_t &tm, int64_t &tn) {
    const int64_t outer = raster_n ? tiles_m : tiles_n;
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
    pdl_wait();  // set-up done; the previous kernel of the stream has completed
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ producer
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            bool rev = false;  // this tile's k-blocks last to first (alternates per tile when snake)
            for (int64_t tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, rev = args.snake && !rev) {
                int64_t tm, tn;
                mx_tile_coords(tile, tiles_m, tiles_n, args.raster_n, args.group, tm, tn);
                const bool sfb1 = 2 * tn + 1 < args.sfb_rows;
                for (int kq = 0; kq < num_kb; kq++) {
                    const int kb = rev ? num_kb - 1 - kq : kq;
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
            const SDesc desc0 = sdesc_k_sw128_split(smem_u32(smem));  // stage 0's A tile
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
                    const uint32_t lo_a = desc0.lo + (uint32_t)s * (AB_BYTES >> 4);
                    const uint32_t lo_b = lo_a + (A_BYTES >> 4);
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
                        umma_mxf8f6f4(tmem_base, sdesc_join(lo_a + 2 * kk, desc0.hi), sdesc_join(lo_b + 2 * kk, desc0.hi),
                                      idesc, t_sfa, t_sfb, (kb | kk) != 0);
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
            mx_tile_coords(tile, tiles_m, tiles_n, args.raster_n, args.group, tm, tn);
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
                            uint8_t *row_s, uint8_t *col_q, uint8_t *col_s, float *dbias, void *workspace,
                            size_t workspace_bytes, fp8dl_stream_t stream) {
    FP8DL_NVTX("mxfp8_quantize");
    FP8DL_CHECK_ARG(x != nullptr, "x is NULL");
    FP8DL_CHECK_ARG(x_dtype == FP8DL_F32 || x_dtype == FP8DL_BF16, "x_dtype must be FP8DL_F32 or FP8DL_BF16");
    FP8DL_CHECK_ARG((row_q == nullptr) == (row_s == nullptr), "row_q and row_s must both be given or both NULL");
    FP8DL_CHECK_ARG((col_q == nullptr) == (col_s == nullptr), "col_q and col_s must both be given or both NULL");
    FP8DL_CHECK_ARG(row_q || col_q, "nothing to compute: all outputs are NULL");
    if (!dim_ok(rows, 32) || !dim_ok(cols, 32))
        return fail(FP8DL_ERR_SHAPE, "rows (%lld) and cols (%lld) must be positive multiples of 32",
                    (long long)rows, (long long)cols);
    if (!aligned16(x) || !aligned16(row_q) || !aligned16(col_q) || !aligned16(dbias))
        return fail(FP8DL_ERR_ALIGN, "x, row_q, col_q and dbias must be 16-byte aligned");
    const int64_t row_tiles = (rows + 127) / 128;
    if (dbias) {
        const size_t need = (size_t)row_tiles * (size_t)cols * sizeof(float);
        if (!workspace || workspace_bytes < need)
            return fail(FP8DL_ERR_WORKSPACE, "mxfp8_quantize: dbias needs a workspace of %zu bytes (got %zu)", need,
                        workspace ? workspace_bytes : (size_t)0);
        if (!aligned16(workspace)) return fail(FP8DL_ERR_ALIGN, "workspace must be 16-byte aligned");
    }
    float *ws = dbias ? static_cast<float *>(workspace) : nullptr;
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    const int64_t tiles = row_tiles * ((cols + 127) / 128);
    const int64_t max_ctas = (int64_t)sms * 2;
    const unsigned grid = (unsigned)(tiles < max_ctas ? tiles : max_ctas);
    const size_t smem = (size_t)MQ_STAGES * 128 * 128 * (x_dtype == FP8DL_BF16 ? 2 : 4);
    static std::atomic<bool> attr[64];
    if (!attr[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(init_mutex());
        if (!attr[dev].load(std::memory_order_relaxed)) {
            cudaError_t e = cudaSuccess;
            for (const void *k : {(const void *)mxfp8_quantize_kernel<FP8DL_BF16, false>,
                                  (const void *)mxfp8_quantize_kernel<FP8DL_BF16, true>})
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MQ_STAGES * 128 * 128 * 2);
            for (const void *k : {(const void *)mxfp8_quantize_kernel<FP8DL_F32, false>,
                                  (const void *)mxfp8_quantize_kernel<FP8DL_F32, true>})
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MQ_STAGES * 128 * 128 * 4);
            if (e != cudaSuccess) return fail(FP8DL_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            attr[dev].store(true, std::memory_order_release);
        }
    }
    const cudaStream_t st = (cudaStream_t)stream;
    const bool pdl = short_call_bytes((double)rows * cols * (x_dtype == FP8DL_BF16 ? 4 : 6));
    if (x_dtype == FP8DL_BF16) {
        if (ws)
            (void)launch_kernel(mxfp8_quantize_kernel<FP8DL_BF16, true>, grid, MQ_THREADS, smem, st, 0, pdl, x, rows, cols, row_q, row_s, col_q,
                                                                                  col_s, ws);
        else
            (void)launch_kernel(mxfp8_quantize_kernel<FP8DL_BF16, false>, grid, MQ_THREADS, smem, st, 0, pdl, x, rows, cols, row_q, row_s, col_q,
                                                                                   col_s, nullptr);
    } else {
        if (ws)
            (void)launch_kernel(mxfp8_quantize_kernel<FP8DL_F32, true>, grid, MQ_THREADS, smem, st, 0, pdl, x, rows, cols, row_q, row_s, col_q,
                                                                                 col_s, ws);
        else
            (void)launch_kernel(mxfp8_quantize_kernel<FP8DL_F32, false>, grid, MQ_THREADS, smem, st, 0, pdl, x, rows, cols, row_q, row_s, col_q,
                                                                                  col_s, nullptr);
    }
    note_launch();
    FP8DL_TRY(check_launch("mxfp8_quantize"));
    if (dbias) {
        colsum_reduce(ws, row_tiles, cols, dbias, (cudaStream_t)stream, pdl);
        FP8DL_TRY(check_launch("mxfp8_quantize(dbias reduce)"));
    }
    if (row_s) launch_sf_pad(row_s, rows, cols / 32, (cudaStream_t)stream, pdl);
    if (col_s) launch_sf_pad(col_s, cols, rows / 32, (cudaStream_t)stream, pdl);
    return check_launch("mxfp8_quantize(scale padding)");
}

fp8dl_status mxfp8_gemm(const uint8_t *A, const uint8_t *A_s, const uint8_t *B, const uint8_t *B_s, int64_t M,
                        int64_t N, int64_t K, const void *bias, int32_t bias_dtype, void *D, int32_t d_dtype,
                        int32_t *dev_status, fp8dl_stream_t stream) {
    FP8DL_NVTX("mxfp8_gemm");
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
    pick_raster(M, N, K, mx::BM, mx::BN, args.raster_n, args.group);
    static std::atomic<bool> attr_set[64];
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(init_mutex());
        if (!attr_set[dev].load(std::memory_order_relaxed)) {
            cudaError_t e =
                cudaFuncSetAttribute(mxfp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mx::SMEM_BYTES);
            if (e != cudaSuccess) return fail(FP8DL_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            attr_set[dev].store(true, std::memory_order_release);
        }
    }
    const int64_t tiles = ((M + mx::BM - 1) / mx::BM) * ((N + mx::BN - 1) / mx::BN);
    const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
    args.snake = pick_snake(tiles, grid, K);
    const bool pdl = short_call_flops(2.0 * (double)M * (double)N * (double)K);
    (void)launch_kernel(mxfp8_gemm_kernel, grid, mx::THREADS, mx::SMEM_BYTES, (cudaStream_t)stream, 0, pdl, ta, tb, args);
    note_launch();
    return check_launch("mxfp8_gemm");
}

}  // extern "C"
