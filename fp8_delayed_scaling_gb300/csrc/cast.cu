// cast.cu — fused FP8 cast + amax + transposed copy (+ bias gradient).
//
// "FP8 低精度训练：Transformer Engine 简析", §三.3 "FP8框架TE计算流程": before
// fp8_gemm the input and weight are cast to FP8 with the scale stored in
// fp8_meta and the cast writes the tensor's amax into the amax history; §三.1:
// delayed scaling knows the scale before the cast, so cast and amax happen in
// one pass over the high-precision tensor (no extra HBM round trip, unlike
// just-in-time scaling).  The transposed copy feeds the backward GEMMs, which
// need the other operand orientation (every GEMM here is K-contiguous).
//
// Design (HBM-bound; one read of x, one write per requested output):
//   tile = 128 rows x 128 cols, 256 threads, persistent grid-stride loop.
//   phase 1: thread (rb, cb) loads rows 4rb..4rb+3, cols 16cb..16cb+15 with
//            16-byte loads, converts with cvt.rn.satfinite, stores 16-byte
//            row-major codes, and stages them in shared memory (16-byte chunks
//            XOR-swizzled by row so both phases are bank-conflict free).
//   phase 2: thread (w, 16-row half) gathers 16 rows x 4 cols, transposes 4x4
//            byte blocks with prmt, and stores 16 bytes per transposed row
//            (two neighbouring threads fill one 32-byte sector).
//   amax: |x| max per thread -> warp shuffle -> one atomicMax per CTA.
//   dbias: per-tile column sums (fp32, fixed order) to a workspace row per
//          128-row tile, then a second kernel sums the tile rows in order.
#include <cuda_bf16.h>

#include "common.cuh"

namespace fp8dl {

constexpr int CT_ROWS = 128, CT_COLS = 128, CT_THREADS = 256;

template <int XKIND>  // 0 = fp32, 1 = bf16
struct RowSeg16;      // 16 consecutive elements of one row

template <>
struct RowSeg16<FP8DL_BF16> {
    uint4 v[2];
    __device__ __forceinline__ void load(const void *p) {
        const uint4 *q = reinterpret_cast<const uint4 *>(p);
        v[0] = ldg_stream(q);
        v[1] = ldg_stream(q + 1);
    }
    __device__ __forceinline__ float get(int j) const {
        const uint32_t w = reinterpret_cast<const uint32_t *>(v)[j >> 1];
        return (j & 1) ? bf16_hi(w) : bf16_lo(w);
    }
};

template <>
struct RowSeg16<FP8DL_F32> {
    uint4 v[4];
    __device__ __forceinline__ void load(const void *p) {
        const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
        for (int i = 0; i < 4; i++) v[i] = ldg_stream(q + i);
    }
    __device__ __forceinline__ float get(int j) const {
        return __uint_as_float(reinterpret_cast<const uint32_t *>(v)[j]);
    }
};

// Byte offset of 16-byte chunk `chunk` of staged row `r` (rows are 128 bytes).
__device__ __forceinline__ int stage_off(int r, int chunk) { return r * CT_COLS + ((chunk ^ ((r >> 2) & 7)) << 4); }

// Element operation fused in front of the cast.
enum CastOp { OP_NONE = 0, OP_GELU = 1, OP_DGELU = 2, OP_LAYERNORM = 3 };

// Extra inputs of the element operation: h for dGELU; per-row mean/rsigma and
// per-column gamma/beta (bf16) for LayerNorm.
struct OpArgs {
    const void *aux;
    const float *mu, *rs;
    const uint16_t *gamma, *beta;
};

// Column sums (csum: this thread's 16 columns as pairs, in the tile's phase-1 layout) added
// over the CTA's threads in a fixed order (lanes l, l+8, l+16, l+24 of a warp, then the eight
// warps) and written to ws_row[0 .. 128) (columns c0 .. c0 + 127; none beyond cols).  Every
// thread calls it; it holds two CTA barriers.
__device__ __forceinline__ void colsum_flush(float2 (&csum)[8], float (*red)[CT_COLS], float *ws_row, int64_t c0,
                                             int64_t cols) {
    const int t = threadIdx.x, lane = t & 31, wi = t >> 5, cb = t & 7;
#pragma unroll
    for (int k = 0; k < 8; k++) {
#pragma unroll
        for (int o = 8; o <= 16; o <<= 1) {
            const float2 p = make_float2(__shfl_xor_sync(0xffffffffu, csum[k].x, o),
                                         __shfl_xor_sync(0xffffffffu, csum[k].y, o));
            csum[k] = __fadd2_rn(csum[k], p);
        }
    }
    if (lane < 8) {
        float4 *dst = reinterpret_cast<float4 *>(&red[wi][16 * cb]);
#pragma unroll
        for (int j = 0; j < 4; j++)
            dst[j] = make_float4(csum[2 * j].x, csum[2 * j].y, csum[2 * j + 1].x, csum[2 * j + 1].y);
    }
    __syncthreads();
    if (t < CT_COLS && c0 + t < cols) {
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < CT_THREADS / 32; k++) s += red[k][t];
        ws_row[t] = s;
    }
    __syncthreads();
}

// One 128 x 128 tile of the cast; every thread of the CTA calls it with the same tile.
// amax: the calling thread's running max of |x|.
template <int XKIND, int FMT, int OP, bool ACC>
__device__ __forceinline__ void cast_tile(const void *__restrict__ x, const OpArgs &op, int64_t rows, int64_t cols,
                                          int64_t tile, float scale, uint8_t *__restrict__ out,
                                          uint8_t *__restrict__ out_t, float *__restrict__ ws,
                                          uint16_t *__restrict__ pre_out, uint8_t *stage, float (*red)[CT_COLS],
                                          float &amax, float2 *accsm) {
    constexpr int ESZ = XKIND == FP8DL_BF16 ? 2 : 4;
    const int t = threadIdx.x;
    const int cb = t & 7, rb = t >> 3;                               // phase 1
    const int lane = t & 31, wi = t >> 5;                            // phase 2
    const int p2_h = lane & 1, p2_w = (wi & 1) * 16 + (lane >> 1), p2_rg = wi >> 1;
    const int64_t tiles_c = (cols + CT_COLS - 1) / CT_COLS;
    const int64_t r0 = (tile / tiles_c) * CT_ROWS, c0 = (tile % tiles_c) * CT_COLS;
    const bool p1_ok = (r0 + 4 * rb < rows) && (c0 + 16 * cb < cols);
    float2 csum[8];  // column sums for dbias: columns 16cb + 2k, +1 in csum[k]
#pragma unroll
    for (int k = 0; k < 8; k++) csum[k] = make_float2(0.0f, 0.0f);
    uint32_t amax2 = 0;  // bf16x2 running |x| maxima (plain bf16 casts)
    if (p1_ok) {
        RowSeg16<XKIND> seg[4];
        RowSeg16<XKIND> hseg[OP == OP_DGELU ? 4 : 1];
        const int64_t eoff = (r0 + 4 * rb) * cols + c0 + 16 * cb;
        const char *base = static_cast<const char *>(x) + eoff * ESZ;
#pragma unroll
        for (int i = 0; i < 4; i++) seg[i].load(base + i * cols * ESZ);
        float ln_mu[4], ln_rs[4];
        uint32_t ln_g[8], ln_b[8];
        if (OP == OP_LAYERNORM) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                ln_mu[i] = __ldg(op.mu + r0 + 4 * rb + i);
                ln_rs[i] = __ldg(op.rs + r0 + 4 * rb + i);
            }
            const uint4 g0 = __ldg(reinterpret_cast<const uint4 *>(op.gamma + c0 + 16 * cb));
            const uint4 g1 = __ldg(reinterpret_cast<const uint4 *>(op.gamma + c0 + 16 * cb + 8));
            const uint4 b0 = __ldg(reinterpret_cast<const uint4 *>(op.beta + c0 + 16 * cb));
            const uint4 b1 = __ldg(reinterpret_cast<const uint4 *>(op.beta + c0 + 16 * cb + 8));
            ln_g[0] = g0.x; ln_g[1] = g0.y; ln_g[2] = g0.z; ln_g[3] = g0.w;
            ln_g[4] = g1.x; ln_g[5] = g1.y; ln_g[6] = g1.z; ln_g[7] = g1.w;
            ln_b[0] = b0.x; ln_b[1] = b0.y; ln_b[2] = b0.z; ln_b[3] = b0.w;
            ln_b[4] = b1.x; ln_b[5] = b1.y; ln_b[6] = b1.z; ln_b[7] = b1.w;
        }
        if (OP == OP_DGELU) {
            const char *hbase = static_cast<const char *>(op.aux) + eoff * ESZ;
#pragma unroll
            for (int i = 0; i < 4; i++) hseg[OP == OP_DGELU ? i : 0].load(hbase + i * cols * ESZ);
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t w[4];
            const int r = 4 * rb + i;
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {  // two halves of 8 elements
                if constexpr (XKIND == FP8DL_BF16 && OP == OP_NONE) {
                    // plain bf16 cast, two elements per instruction: |x| maxima on the bf16x2
                    // words, fp32 products x * scale, column sums
                    const uint4 q = seg[i].v[hh];
                    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
                    const float2 sc2 = make_float2(scale, scale);
                    float2 f[4];
#pragma unroll
                    for (int p = 0; p < 4; p++) {
                        amax2 = bf16x2_absmax(amax2, qw[p]);
                        f[p] = make_float2(bf16_lo(qw[p]), bf16_hi(qw[p]));
                        if (ws) csum[4 * hh + p] = __fadd2_rn(csum[4 * hh + p], f[p]);
                        f[p] = __fmul2_rn(f[p], sc2);
                    }
                    w[2 * hh] = pack4<FMT>(f[0].x, f[0].y, f[1].x, f[1].y);
                    w[2 * hh + 1] = pack4<FMT>(f[2].x, f[2].y, f[3].x, f[3].y);
                } else {
                    float v[8];
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        float xv = seg[i].get(8 * hh + j);
                        if (OP == OP_GELU) xv = gelu_bf16(xv);
                        if (OP == OP_DGELU) xv = dgelu_bf16(xv, hseg[OP == OP_DGELU ? i : 0].get(8 * hh + j));
                        if (OP == OP_LAYERNORM) {
                            const int k = 8 * hh + j;  // y = bf16((x - mu) * rs * gamma + beta)
                            const float gk = (k & 1) ? bf16_hi(ln_g[k >> 1]) : bf16_lo(ln_g[k >> 1]);
                            const float bk = (k & 1) ? bf16_hi(ln_b[k >> 1]) : bf16_lo(ln_b[k >> 1]);
                            xv = bf16_round(fmaf((xv - ln_mu[i]) * ln_rs[i], gk, bk));
                        }
                        v[j] = xv;
                        amax = fmaxf(amax, fabsf(xv));
                        if (OP == OP_NONE || OP == OP_DGELU) {  // dbias only there
                            if (j & 1)
                                csum[4 * hh + (j >> 1)].y += xv;
                            else
                                csum[4 * hh + (j >> 1)].x += xv;
                        }
                    }
                    w[2 * hh] = pack4<FMT>(__fmul_rn(v[0], scale), __fmul_rn(v[1], scale), __fmul_rn(v[2], scale),
                                           __fmul_rn(v[3], scale));
                    w[2 * hh + 1] = pack4<FMT>(__fmul_rn(v[4], scale), __fmul_rn(v[5], scale),
                                               __fmul_rn(v[6], scale), __fmul_rn(v[7], scale));
                    if (OP != OP_NONE && pre_out) {
                        uint32_t pw[4];
#pragma unroll
                        for (int p = 0; p < 4; p++) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * p], v[2 * p + 1]);
                            pw[p] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(pre_out + (r0 + r) * cols + c0 + 16 * cb + 8 * hh) =
                            make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    }
                }
            }
            const uint4 codes = make_uint4(w[0], w[1], w[2], w[3]);
            if (out) *reinterpret_cast<uint4 *>(out + (r0 + r) * cols + c0 + 16 * cb) = codes;
            if (out_t) *reinterpret_cast<uint4 *>(stage + stage_off(r, cb)) = codes;
        }
    }
    if constexpr (XKIND == FP8DL_BF16 && OP == OP_NONE)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(amax2)), fabsf(bf16_hi(amax2))));
    // ACC: the CTA's running column sums in shared memory (accsm[k][thread]), flushed by the
    // caller after its last tile; else this tile writes its own ws row
    if constexpr (ACC) {
        if (ws) {
#pragma unroll
            for (int k = 0; k < 8; k++)
                accsm[k * CT_THREADS + t] = __fadd2_rn(accsm[k * CT_THREADS + t], csum[k]);
        }
    }
    const bool wsf = !ACC && ws;  // this tile's column sums go to its own ws row (after phase 2)
    if (out_t) __syncthreads();
    if (out_t) {
        const int rl = 32 * p2_rg + 16 * p2_h;  // first of this thread's 16 rows within the tile
        if (r0 + rl < rows && c0 + 4 * p2_w < cols) {
            uint32_t col[4][4];  // col[j][g]: rows rl+4g..rl+4g+3 of column 4*p2_w+j
#pragma unroll
            for (int g = 0; g < 4; g++) {
                uint32_t W[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int r = rl + 4 * g + k;
                    W[k] = *reinterpret_cast<const uint32_t *>(stage + stage_off(r, p2_w >> 2) + 4 * (p2_w & 3));
                }
                const uint32_t t0 = __byte_perm(W[0], W[1], 0x5140), t1 = __byte_perm(W[2], W[3], 0x5140);
                const uint32_t t2 = __byte_perm(W[0], W[1], 0x7362), t3 = __byte_perm(W[2], W[3], 0x7362);
                col[0][g] = __byte_perm(t0, t1, 0x5410);
                col[1][g] = __byte_perm(t0, t1, 0x7632);
                col[2][g] = __byte_perm(t2, t3, 0x5410);
                col[3][g] = __byte_perm(t2, t3, 0x7632);
            }
#pragma unroll
            for (int j = 0; j < 4; j++)
                *reinterpret_cast<uint4 *>(out_t + (c0 + 4 * p2_w + j) * rows + r0 + rl) =
                    make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]);
        }
    }
    if (out_t) __syncthreads();
    if (wsf) colsum_flush(csum, red, ws + (r0 / CT_ROWS) * cols + c0, c0, cols);
}

// The CTA's largest |x| max-ed into *amax_p; every thread calls it (wmax: CT_THREADS / 32 floats).
__device__ __forceinline__ void cta_amax_flush(float amax, float *amax_p, float *wmax) {
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const float m = warp_max(amax);
    if (lane == 0) wmax[wi] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = wmax[0];
        for (int k = 1; k < CT_THREADS / 32; k++) mm = fmaxf(mm, wmax[k]);
        atomic_max_nonneg(amax_p, mm);
    }
    __syncthreads();  // wmax is free again
}

template <int XKIND, int FMT, int OP, bool ACC>
__global__ void __launch_bounds__(CT_THREADS, OP == OP_LAYERNORM ? 2 : OP != OP_NONE ? 3 : (XKIND == FP8DL_BF16 ? 4 : 2))
    cast_kernel(const void *__restrict__ x, const OpArgs op, int64_t rows, int64_t cols,
                const float *__restrict__ scale_p, uint8_t *__restrict__ out, uint8_t *__restrict__ out_t,
                float *__restrict__ amax_p, float *__restrict__ ws, uint16_t *__restrict__ pre_out) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    __shared__ __align__(16) uint8_t stage[CT_ROWS * CT_COLS];
    __shared__ __align__(16) float red[CT_THREADS / 32][CT_COLS];  // per-warp column partials (dbias)
    __shared__ __align__(16) float2 accsm[ACC ? 8 * CT_THREADS : 1];  // running column sums (ACC)
    __shared__ float wmax[CT_THREADS / 32];
    const float scale = out || out_t ? __ldg(scale_p) : 1.0f;
    const int64_t tiles_c = (cols + CT_COLS - 1) / CT_COLS, tiles = ((rows + CT_ROWS - 1) / CT_ROWS) * tiles_c;
    float amax = 0.0f;
    // ACC: the grid is a multiple of tiles_c, so every tile of this CTA lies in column block
    // blockIdx.x % tiles_c; its column sums gather in accsm and go to ws row blockIdx.x / tiles_c
    // once.  Otherwise every tile writes its own ws row.
    const bool acc = ACC && ws;
    if (acc) {
#pragma unroll
        for (int k = 0; k < 8; k++) accsm[k * CT_THREADS + threadIdx.x] = make_float2(0.0f, 0.0f);
    }
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x)
        cast_tile<XKIND, FMT, OP, ACC>(x, op, rows, cols, tile, scale, out, out_t, ws, pre_out, stage, red, amax,
                                       accsm);
    if (acc) {
        float2 csum[8];
#pragma unroll
        for (int k = 0; k < 8; k++) csum[k] = accsm[k * CT_THREADS + threadIdx.x];
        const int64_t c0 = (blockIdx.x % tiles_c) * CT_COLS;
        colsum_flush(csum, red, ws + (blockIdx.x / tiles_c) * cols + c0, c0, cols);
    }
    if (amax_p) cta_amax_flush(amax, amax_p, wmax);
}

// Several tensors cast in one launch: their tiles are numbered one tensor after the
// other, and each CTA walks tiles blockIdx.x, + gridDim.x, ... of the whole set.  A
// CTA's tiles reach the tensors in order, so it flushes its amax once per tensor.
constexpr int CAST_MULTI_MAX = 8;
struct CastMultiArgs {
    int n;
    const void *x[CAST_MULTI_MAX];
    int64_t rows[CAST_MULTI_MAX], cols[CAST_MULTI_MAX];
    const float *scale[CAST_MULTI_MAX];
    uint8_t *out[CAST_MULTI_MAX], *out_t[CAST_MULTI_MAX];
    float *amax[CAST_MULTI_MAX];
    float *scale_inv_out[CAST_MULTI_MAX];
    int64_t tile_end[CAST_MULTI_MAX];  // tiles of tensors 0 .. k together
};

template <int XKIND, int FMT>
__global__ void __launch_bounds__(CT_THREADS, XKIND == FP8DL_BF16 ? 4 : 2)
    cast_multi_kernel(const __grid_constant__ CastMultiArgs a) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    __shared__ __align__(16) uint8_t stage[CT_ROWS * CT_COLS];
    __shared__ __align__(16) float red[CT_THREADS / 32][CT_COLS];  // unused: no bias gradients here
    __shared__ float wmax[CT_THREADS / 32];
    const int64_t tiles = a.tile_end[a.n - 1];
    int item = 0;
    float amax = 0.0f;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        int k = item;
        while (tile >= a.tile_end[k]) k++;
        if (k != item) {  // the same for every thread of the CTA
            if (a.amax[item]) cta_amax_flush(amax, a.amax[item], wmax);
            amax = 0.0f;
            item = k;
        }
        const int64_t first = item ? a.tile_end[item - 1] : 0;
        const float scale = (a.out[item] || a.out_t[item]) ? __ldg(a.scale[item]) : 1.0f;
        cast_tile<XKIND, FMT, OP_NONE, false>(a.x[item], OpArgs{}, a.rows[item], a.cols[item], tile - first, scale,
                                       a.out[item], a.out_t[item], nullptr, nullptr, stage, red, amax, nullptr);
    }
    if (a.amax[item]) cta_amax_flush(amax, a.amax[item], wmax);
}

// The decode factors fl32(1 / scale) of the tensors of a grouped cast that ask for one.
__global__ void scale_inv_multi_kernel(const __grid_constant__ CastMultiArgs a) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    const int k = threadIdx.x;
    if (k < a.n && a.scale_inv_out[k]) *a.scale_inv_out[k] = __frcp_rn(*a.scale[k]);
}

// dbias[c] = sum over row tiles of ws[tile][c], in a fixed order: CTA = 32
// columns x 8 warps; warp w sums tiles w, w+8, ... (lane = column), then the 8
// partials are added in warp order.
constexpr int RED_COLS = 32, RED_WARPS = 8;

__global__ void __launch_bounds__(RED_COLS *RED_WARPS) colsum_reduce_kernel(const float *__restrict__ ws,
                                                                            int64_t n_tiles, int64_t cols,
                                                                            float *__restrict__ dbias) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    __shared__ float part[RED_WARPS][RED_COLS];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t c = blockIdx.x * (int64_t)RED_COLS + lane;
    float s = 0.0f;
    if (c < cols) {
        // 16 loads in flight, then their sums in the same order as one at a time
        int64_t k = w;
        for (; k + 15 * RED_WARPS < n_tiles; k += 16 * RED_WARPS) {
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; u++) v[u] = ws[(k + u * RED_WARPS) * cols + c];
#pragma unroll
            for (int u = 0; u < 16; u++) s += v[u];
        }
        for (; k < n_tiles; k += RED_WARPS) s += ws[k * cols + c];
    }
    part[w][lane] = s;
    __syncthreads();
    if (w == 0 && c < cols) {
        float t = 0.0f;
#pragma unroll
        for (int k = 0; k < RED_WARPS; k++) t += part[k][lane];
        dbias[c] = t;
    }
}

static void launch_colsum_reduce(const float *ws, int64_t n_tiles, int64_t cols, float *dbias, cudaStream_t st,
                                 bool pdl) {
    (void)launch_kernel(colsum_reduce_kernel, (unsigned)((cols + RED_COLS - 1) / RED_COLS), RED_COLS * RED_WARPS, 0, st, 0, pdl, ws, n_tiles,
                                                                                                       cols, dbias);
    note_launch();
}

void colsum_reduce(const float *ws, int64_t n_rows, int64_t cols, float *dbias, cudaStream_t st, bool pdl) {
    launch_colsum_reduce(ws, n_rows, cols, dbias, st, pdl);
}

// Grid of a tiled cast launch: no more CTAs than fit on the GPU at once.  Every CTA is then
// resident from the start and walks tiles blockIdx.x, + gridDim.x, ..., so the CTAs' tile
// counts differ by at most one.  (With more CTAs than slots, CTAs of 3 and 4 tiles queue
// behind each other and the last slots finish up to two tiles after the average.)
// per_sm caches the kernel's resident CTAs per SM (the same on every sm_103 device).
static dim3 resident_grid(const void *kernel, std::atomic<int> &per_sm, int64_t tiles, int sms) {
    int occ = per_sm.load(std::memory_order_acquire);
    if (occ == 0) {
        std::lock_guard<std::mutex> lock(init_mutex());
        occ = per_sm.load(std::memory_order_relaxed);
        if (occ == 0) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, CT_THREADS, 0) != cudaSuccess || n < 1) {
                cudaGetLastError();
                n = 1;
            }
            occ = n;
            per_sm.store(occ, std::memory_order_release);
        }
    }
    const int64_t slots = (int64_t)sms * occ;
    return dim3((unsigned)(tiles < slots ? tiles : slots));
}

template <int XKIND, int FMT, int OP, bool ACC = false>
static dim3 cast_grid(int64_t tiles, int sms) {
    static std::atomic<int> per_sm{0};
    return resident_grid((const void *)cast_kernel<XKIND, FMT, OP, ACC>, per_sm, tiles, sms);
}

// A cast with column sums (ws != NULL) runs the running-sum variant when its grid can be a
// multiple of the column-tile count: every CTA then stays in one column block and writes one
// ws row.  Returns the ws rows the column-sum reduction adds.
template <int XKIND, int FMT, int OP>
static int64_t launch_cast_op(int64_t tiles, int sms, cudaStream_t st, const void *x, const OpArgs &op, int64_t rows,
                              int64_t cols, const float *scale, uint8_t *out, uint8_t *out_t, float *amax, float *ws,
                              uint16_t *pre_out, bool pdl) {
    const int64_t tiles_c = (cols + CT_COLS - 1) / CT_COLS;
    if (ws) {
        dim3 grid = cast_grid<XKIND, FMT, OP, true>(tiles, sms);
        if ((int64_t)grid.x >= tiles_c) {
            grid.x -= (unsigned)((int64_t)grid.x % tiles_c);
            (void)launch_kernel(cast_kernel<XKIND, FMT, OP, true>, grid, CT_THREADS, 0, st, 0, pdl, x, op, rows, cols,
                                scale, out, out_t, amax, ws, pre_out);
            note_launch();
            return (int64_t)grid.x / tiles_c;
        }
    }
    (void)launch_kernel(cast_kernel<XKIND, FMT, OP, false>, cast_grid<XKIND, FMT, OP, false>(tiles, sms), CT_THREADS, 0,
                        st, 0, pdl, x, op, rows, cols, scale, out, out_t, amax, ws, pre_out);
    note_launch();
    return (rows + CT_ROWS - 1) / CT_ROWS;
}

template <int XKIND, int FMT>
static int64_t launch_cast(int64_t tiles, int sms, cudaStream_t st, const void *x, int64_t rows, int64_t cols,
                           const float *scale, uint8_t *out, uint8_t *out_t, float *amax, float *ws, bool pdl) {
    return launch_cast_op<XKIND, FMT, OP_NONE>(tiles, sms, st, x, OpArgs{}, rows, cols, scale, out, out_t, amax, ws,
                                               nullptr, pdl);
}

template <int OP>
static int64_t launch_op_cast(int64_t tiles, int sms, cudaStream_t st, int fmt, const void *x, const OpArgs &op,
                              int64_t rows, int64_t cols, const float *scale, uint8_t *out, uint8_t *out_t,
                              float *amax, float *ws, uint16_t *pre_out, bool pdl) {
    if (fmt == FP8DL_E4M3)
        return launch_cast_op<FP8DL_BF16, FP8DL_E4M3, OP>(tiles, sms, st, x, op, rows, cols, scale, out, out_t, amax, ws,
                                                          pre_out, pdl);
    return launch_cast_op<FP8DL_BF16, FP8DL_E5M2, OP>(tiles, sms, st, x, op, rows, cols, scale, out, out_t, amax, ws,
                                                      pre_out, pdl);
}

// LayerNorm + cast over 128 x 128 tiles, given the per-row statistics (used by
// fp8_layernorm_cast after its row-statistics pass).
fp8dl_status launch_layernorm_tile_cast(const void *x, const float *mu, const float *rs, const void *gamma,
                                        const void *beta, int64_t rows, int64_t cols, int fmt, const float *scale,
                                        uint8_t *out, uint8_t *out_t, float *amax, void *y, int sms,
                                        cudaStream_t st, bool pdl) {
    const int64_t tiles = ((rows + CT_ROWS - 1) / CT_ROWS) * ((cols + CT_COLS - 1) / CT_COLS);
    OpArgs op{nullptr, mu, rs, static_cast<const uint16_t *>(gamma), static_cast<const uint16_t *>(beta)};
    launch_op_cast<OP_LAYERNORM>(tiles, sms, st, fmt, x, op, rows, cols, scale, out, out_t, amax, nullptr,
                                 static_cast<uint16_t *>(y), pdl);
    return check_launch("fp8_layernorm_cast(tiles)");
}

// The decode factor of codes cast at *scale: fl32(1 / scale), the same
// rounding as the scale_inv the scale update stores beside the scale.
__global__ void scale_inv_snapshot_kernel(const float *scale, float *scale_inv) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    if (threadIdx.x == 0) *scale_inv = __frcp_rn(*scale);
}

}  // namespace fp8dl

using namespace fp8dl;

extern "C" {

size_t fp8_cast_workspace_size(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)((rows + CT_ROWS - 1) / CT_ROWS) * (size_t)cols * sizeof(float);
}

fp8dl_status fp8_cast_amax_transpose(const void *x, int32_t x_dtype, int64_t rows, int64_t cols, int32_t out_dtype,
                                     const float *scale, uint8_t *out, uint8_t *out_t, float *amax,
                                     float *scale_inv_out, float *dbias, void *workspace, size_t workspace_bytes,
                                     fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_cast_amax_transpose");
    FP8DL_CHECK_ARG(x != nullptr, "x is NULL");
    FP8DL_CHECK_ARG(!scale_inv_out || scale != nullptr, "scale_inv_out needs scale");
    FP8DL_CHECK_ARG(x_dtype == FP8DL_F32 || x_dtype == FP8DL_BF16, "x_dtype must be FP8DL_F32 or FP8DL_BF16");
    FP8DL_CHECK_ARG(out_dtype == FP8DL_E4M3 || out_dtype == FP8DL_E5M2, "out_dtype must be E4M3 or E5M2");
    FP8DL_CHECK_ARG(!(out || out_t) || scale != nullptr, "scale is NULL but an FP8 output was requested");
    FP8DL_CHECK_ARG(out || out_t || amax || dbias, "nothing to compute: all outputs are NULL");
    if (!dim_ok(rows, 16) || !dim_ok(cols, 16))
        return fail(FP8DL_ERR_SHAPE, "rows (%lld) and cols (%lld) must be positive multiples of 16",
                    (long long)rows, (long long)cols);
    if (!aligned16(x) || !aligned16(out) || !aligned16(out_t) || !aligned16(dbias))
        return fail(FP8DL_ERR_ALIGN, "x, out, out_t and dbias must be 16-byte aligned");
    if (dbias) {
        if (!workspace || workspace_bytes < fp8_cast_workspace_size(rows, cols))
            return fail(FP8DL_ERR_WORKSPACE, "dbias needs a workspace of %zu bytes (got %zu)",
                        fp8_cast_workspace_size(rows, cols), workspace ? workspace_bytes : (size_t)0);
        if (!aligned16(workspace)) return fail(FP8DL_ERR_ALIGN, "workspace must be 16-byte aligned");
    }
    int sms = 0;
    FP8DL_TRY(current_device(nullptr, &sms));
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t tiles = ((rows + CT_ROWS - 1) / CT_ROWS) * ((cols + CT_COLS - 1) / CT_COLS);
    float *ws = dbias ? static_cast<float *>(workspace) : nullptr;
    const bool pdl = short_call_bytes((double)rows * cols * (x_dtype == FP8DL_BF16 ? 4 : 6));
    int64_t ws_rows = 0;  // ws rows the column-sum reduction adds
    if (x_dtype == FP8DL_BF16) {
        if (out_dtype == FP8DL_E4M3)
            ws_rows = launch_cast<FP8DL_BF16, FP8DL_E4M3>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
        else
            ws_rows = launch_cast<FP8DL_BF16, FP8DL_E5M2>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
    } else {
        if (out_dtype == FP8DL_E4M3)
            ws_rows = launch_cast<FP8DL_F32, FP8DL_E4M3>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
        else
            ws_rows = launch_cast<FP8DL_F32, FP8DL_E5M2>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
    }
    FP8DL_TRY(check_launch("fp8_cast_amax_transpose"));
    if (dbias) {
        launch_colsum_reduce(ws, ws_rows, cols, dbias, st, pdl);
        FP8DL_TRY(check_launch("fp8_cast_amax_transpose(dbias reduce)"));
    }
    if (scale_inv_out) {
        (void)launch_kernel(scale_inv_snapshot_kernel, 1, 32, 0, st, 0, pdl, scale, scale_inv_out);
        note_launch();
        FP8DL_TRY(check_launch("fp8_cast_amax_transpose(scale_inv)"));
    }
    return FP8DL_OK;
}

fp8dl_status fp8_cast_amax_transpose_multi(int32_t n, const fp8dl_cast_item *items, int32_t x_dtype,
                                           int32_t out_dtype, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_cast_amax_transpose_multi");
    FP8DL_CHECK_ARG(n >= 1 && n <= CAST_MULTI_MAX, "n (%d) must be in 1..%d", (int)n, CAST_MULTI_MAX);
    FP8DL_CHECK_ARG(items != nullptr, "items is NULL");
    FP8DL_CHECK_ARG(x_dtype == FP8DL_F32 || x_dtype == FP8DL_BF16, "x_dtype must be FP8DL_F32 or FP8DL_BF16");
    FP8DL_CHECK_ARG(out_dtype == FP8DL_E4M3 || out_dtype == FP8DL_E5M2, "out_dtype must be E4M3 or E5M2");
    CastMultiArgs a{};
    a.n = n;
    bool any_inv = false;
    int64_t tiles = 0;
    double bytes = 0.0;
    for (int k = 0; k < n; k++) {
        const fp8dl_cast_item &it = items[k];
        FP8DL_CHECK_ARG(it.x != nullptr, "item %d: x is NULL", k);
        FP8DL_CHECK_ARG(!(it.out || it.out_t || it.scale_inv_out) || it.scale != nullptr,
                        "item %d: scale is NULL but an output needs it", k);
        FP8DL_CHECK_ARG(it.out || it.out_t || it.amax, "item %d: nothing to compute", k);
        if (!dim_ok(it.rows, 16) || !dim_ok(it.cols, 16))
            return fail(FP8DL_ERR_SHAPE, "item %d: rows (%lld) and cols (%lld) must be positive multiples of 16", k,
                        (long long)it.rows, (long long)it.cols);
        if (!aligned16(it.x) || !aligned16(it.out) || !aligned16(it.out_t))
            return fail(FP8DL_ERR_ALIGN, "item %d: x, out and out_t must be 16-byte aligned", k);
        a.x[k] = it.x;
        a.rows[k] = it.rows;
        a.cols[k] = it.cols;
        a.scale[k] = it.scale;
        a.out[k] = it.out;
        a.out_t[k] = it.out_t;
        a.amax[k] = it.amax;
        a.scale_inv_out[k] = it.scale_inv_out;
        any_inv = any_inv || it.scale_inv_out != nullptr;
        tiles += ((it.rows + CT_ROWS - 1) / CT_ROWS) * ((it.cols + CT_COLS - 1) / CT_COLS);
        a.tile_end[k] = tiles;
        bytes += (double)it.rows * it.cols * (x_dtype == FP8DL_BF16 ? 4 : 6);
    }
    const bool pdl = short_call_bytes(bytes);
    int sms = 0;
    FP8DL_TRY(current_device(nullptr, &sms));
    cudaStream_t st = (cudaStream_t)stream;
    static std::atomic<int> occ[2][2];
    const int xi = x_dtype == FP8DL_BF16, fi = out_dtype == FP8DL_E5M2;
    const void *kern = xi ? (fi ? (const void *)cast_multi_kernel<FP8DL_BF16, FP8DL_E5M2>
                                : (const void *)cast_multi_kernel<FP8DL_BF16, FP8DL_E4M3>)
                          : (fi ? (const void *)cast_multi_kernel<FP8DL_F32, FP8DL_E5M2>
                                : (const void *)cast_multi_kernel<FP8DL_F32, FP8DL_E4M3>);
    const dim3 grid = resident_grid(kern, occ[xi][fi], tiles, sms);
    if (xi) {
        if (fi)
            (void)launch_kernel(cast_multi_kernel<FP8DL_BF16, FP8DL_E5M2>, grid, CT_THREADS, 0, st, 0, pdl, a);
        else
            (void)launch_kernel(cast_multi_kernel<FP8DL_BF16, FP8DL_E4M3>, grid, CT_THREADS, 0, st, 0, pdl, a);
    } else {
        if (fi)
            (void)launch_kernel(cast_multi_kernel<FP8DL_F32, FP8DL_E5M2>, grid, CT_THREADS, 0, st, 0, pdl, a);
        else
            (void)launch_kernel(cast_multi_kernel<FP8DL_F32, FP8DL_E4M3>, grid, CT_THREADS, 0, st, 0, pdl, a);
    }
    note_launch();
    FP8DL_TRY(check_launch("fp8_cast_amax_transpose_multi"));
    if (any_inv) {
        (void)launch_kernel(scale_inv_multi_kernel, 1, 32, 0, st, 0, pdl, a);
        note_launch();
        FP8DL_TRY(check_launch("fp8_cast_amax_transpose_multi(scale_inv)"));
    }
    return FP8DL_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// GELU + cast and dGELU + cast (the LayerNormMLP activation, fused in front of
// the FP8 cast of its output / of the gradient of its input).
// ---------------------------------------------------------------------------
namespace fp8dl {

static fp8dl_status op_cast_common(int op, const void *x, const void *aux, int64_t rows, int64_t cols,
                                   int32_t out_dtype, const float *scale, uint8_t *out, uint8_t *out_t, float *amax,
                                   float *dbias, void *workspace, size_t workspace_bytes, void *pre_out,
                                   fp8dl_stream_t stream, const char *name) {
    FP8DL_CHECK_ARG(x != nullptr && (op != OP_DGELU || aux != nullptr), "%s: input is NULL", name);
    FP8DL_CHECK_ARG(out_dtype == FP8DL_E4M3 || out_dtype == FP8DL_E5M2, "%s: out_dtype must be E4M3 or E5M2", name);
    FP8DL_CHECK_ARG(!(out || out_t) || scale != nullptr, "%s: scale is NULL but an FP8 output was requested", name);
    FP8DL_CHECK_ARG(out || out_t || amax || dbias || pre_out, "%s: nothing to compute", name);
    if (!dim_ok(rows, 16) || !dim_ok(cols, 16))
        return fail(FP8DL_ERR_SHAPE, "%s: rows (%lld) and cols (%lld) must be positive multiples of 16", name,
                    (long long)rows, (long long)cols);
    if (!aligned16(x) || !aligned16(aux) || !aligned16(out) || !aligned16(out_t) || !aligned16(dbias) ||
        !aligned16(pre_out))
        return fail(FP8DL_ERR_ALIGN, "%s: pointers must be 16-byte aligned", name);
    if (dbias) {
        if (!workspace || workspace_bytes < fp8_cast_workspace_size(rows, cols))
            return fail(FP8DL_ERR_WORKSPACE, "%s: dbias needs a workspace of %zu bytes", name,
                        fp8_cast_workspace_size(rows, cols));
        if (!aligned16(workspace)) return fail(FP8DL_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);
    }
    int sms = 0;
    FP8DL_TRY(current_device(nullptr, &sms));
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t tiles = ((rows + CT_ROWS - 1) / CT_ROWS) * ((cols + CT_COLS - 1) / CT_COLS);
    float *ws = dbias ? static_cast<float *>(workspace) : nullptr;
    uint16_t *pre = static_cast<uint16_t *>(pre_out);
    const bool pdl = short_call_bytes((double)rows * cols * (op == OP_DGELU ? 8 : 6));
    int64_t ws_rows = 0;  // ws rows the column-sum reduction adds
    if (op == OP_GELU)
        ws_rows = launch_op_cast<OP_GELU>(tiles, sms, st, out_dtype, x, OpArgs{}, rows, cols, scale, out, out_t, amax, ws, pre,
                                pdl);
    else
        ws_rows = launch_op_cast<OP_DGELU>(tiles, sms, st, out_dtype, x, OpArgs{aux, nullptr, nullptr, nullptr, nullptr}, rows, cols,
                                 scale, out, out_t, amax, ws, pre, pdl);
    FP8DL_TRY(check_launch(name));
    if (dbias) {
        launch_colsum_reduce(ws, ws_rows, cols, dbias, st, pdl);
        FP8DL_TRY(check_launch(name));
    }
    return FP8DL_OK;
}

}  // namespace fp8dl

extern "C" fp8dl_status fp8_gelu_cast(const void *h, int64_t rows, int64_t cols, int32_t out_dtype,
                                      const float *scale, uint8_t *out, uint8_t *out_t, float *amax, void *g,
                                      fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_gelu_cast");
    return fp8dl::op_cast_common(fp8dl::OP_GELU, h, nullptr, rows, cols, out_dtype, scale, out, out_t, amax, nullptr,
                                 nullptr, 0, g, stream, "fp8_gelu_cast");
}

extern "C" fp8dl_status fp8_dgelu_cast(const void *dg, const void *h, int64_t rows, int64_t cols, int32_t out_dtype,
                                       const float *scale, uint8_t *out, uint8_t *out_t, float *amax, float *dbias,
                                       void *workspace, size_t workspace_bytes, void *dh, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_dgelu_cast");
    return fp8dl::op_cast_common(fp8dl::OP_DGELU, dg, h, rows, cols, out_dtype, scale, out, out_t, amax, dbias,
                                 workspace, workspace_bytes, dh, stream, "fp8_dgelu_cast");
}

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory.
//
// Some callers only hand this library their input and output buffers: a
// plugin or custom-op interface with a fixed signature has no workspace
// argument, and a process whose device memory is owned by another allocator
// may not be allowed to call cudaMalloc itself.  Such callers cannot supply
// the bias-gradient workspace of fp8_cast_amax_transpose.  This variant takes
// that workspace from a fixed-size array in the library's own static device
// memory instead; it allocates nothing.
// ---------------------------------------------------------------------------
namespace fp8dl {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB, held on every device that loads the library
static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];
static std::atomic<float *> g_static_scratch_addr[64];  // device address of g_static_scratch, per device index

// The array's name in host code is a host-side stand-in, not a device address:
// look the address up once per device, with that device current.
static fp8dl_status static_scratch_address(int dev, float **out) {
    float *a = g_static_scratch_addr[dev].load(std::memory_order_acquire);
    if (a == nullptr) {
        std::lock_guard<std::mutex> lock(init_mutex());
        a = g_static_scratch_addr[dev].load(std::memory_order_relaxed);
        if (a == nullptr) {
            void *p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
            if (e != cudaSuccess || p == nullptr)
                return fail(FP8DL_ERR_CUDA, "cudaGetSymbolAddress(static scratch) failed: %s", cudaGetErrorString(e));
            a = static_cast<float *>(p);
            g_static_scratch_addr[dev].store(a, std::memory_order_release);
        }
    }
    *out = a;
    return FP8DL_OK;
}

}  // namespace fp8dl

extern "C" fp8dl_status fp8_cast_amax_transpose_noalloc(const void *x, int32_t x_dtype, int64_t rows, int64_t cols,
                                                        int32_t out_dtype, const float *scale, uint8_t *out,
                                                        uint8_t *out_t, float *amax, float *dbias,
                                                        fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_cast_amax_transpose_noalloc");
    FP8DL_CHECK_ARG(x != nullptr, "x is NULL");
    FP8DL_CHECK_ARG(x_dtype == FP8DL_F32 || x_dtype == FP8DL_BF16, "x_dtype must be FP8DL_F32 or FP8DL_BF16");
    FP8DL_CHECK_ARG(out_dtype == FP8DL_E4M3 || out_dtype == FP8DL_E5M2, "out_dtype must be E4M3 or E5M2");
    FP8DL_CHECK_ARG(!(out || out_t) || scale != nullptr, "scale is NULL but an FP8 output was requested");
    FP8DL_CHECK_ARG(out || out_t || amax || dbias, "nothing to compute: all outputs are NULL");
    if (!dim_ok(rows, 16) || !dim_ok(cols, 16))
        return fail(FP8DL_ERR_SHAPE, "rows (%lld) and cols (%lld) must be positive multiples of 16",
                    (long long)rows, (long long)cols);
    if (!aligned16(x) || !aligned16(out) || !aligned16(out_t) || !aligned16(dbias))
        return fail(FP8DL_ERR_ALIGN, "x, out, out_t and dbias must be 16-byte aligned");
    if (dbias && fp8_cast_workspace_size(rows, cols) > kStaticScratchBytes)
        return fail(FP8DL_ERR_WORKSPACE,
                    "fp8_cast_amax_transpose_noalloc: dbias of a %lld x %lld tensor needs %zu bytes of scratch, "
                    "more than the %zu-byte static array (ceil(rows/128) * cols * 4 must be <= %zu)",
                    (long long)rows, (long long)cols, fp8_cast_workspace_size(rows, cols), kStaticScratchBytes,
                    kStaticScratchBytes);
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    float *ws = nullptr;
    if (dbias) FP8DL_TRY(static_scratch_address(dev, &ws));
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t tiles = ((rows + CT_ROWS - 1) / CT_ROWS) * ((cols + CT_COLS - 1) / CT_COLS);
    const bool pdl = short_call_bytes((double)rows * cols * (x_dtype == FP8DL_BF16 ? 4 : 6));
    // The cast's partials and their reduction are enqueued back to back with no other call's
    // launches between them: calls from several host threads on one stream then run one
    // after another on the GPU, each reading its own partials from the shared array.
    static std::mutex scratch_order;
    std::unique_lock<std::mutex> order(scratch_order, std::defer_lock);
    if (dbias) order.lock();
    int64_t ws_rows = 0;  // ws rows the column-sum reduction adds
    if (x_dtype == FP8DL_BF16) {
        if (out_dtype == FP8DL_E4M3)
            ws_rows = launch_cast<FP8DL_BF16, FP8DL_E4M3>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
        else
            ws_rows = launch_cast<FP8DL_BF16, FP8DL_E5M2>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
    } else {
        if (out_dtype == FP8DL_E4M3)
            ws_rows = launch_cast<FP8DL_F32, FP8DL_E4M3>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
        else
            ws_rows = launch_cast<FP8DL_F32, FP8DL_E5M2>(tiles, sms, st, x, rows, cols, scale, out, out_t, amax, ws, pdl);
    }
    FP8DL_TRY(check_launch("fp8_cast_amax_transpose_noalloc"));
    if (dbias) {
        launch_colsum_reduce(ws, ws_rows, cols, dbias, st, pdl);
        FP8DL_TRY(check_launch("fp8_cast_amax_transpose_noalloc(dbias reduce)"));
    }
    return FP8DL_OK;
}
