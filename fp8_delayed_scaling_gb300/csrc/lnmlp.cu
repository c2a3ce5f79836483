// lnmlp.cu — LayerNorm pieces of the LayerNormMLP path: LayerNorm forward fused
// with the FP8 cast of its output, and the LayerNorm backward.
//
// "NVIDIA Transformer Engine 加速训练教程" builds blocks from te.LayerNormMLP
// (LayerNorm -> fc1 -> GELU -> fc2) and mirrors them in plain PyTorch with
// nn.LayerNorm (biased variance).  Under delayed scaling ("FP8 低精度训练：
// Transformer Engine 简析" §三.1/§三.3) the LayerNorm output is what fc1 casts,
// and its scale is known before the LayerNorm runs, so normalisation, bf16
// rounding, the FP8 cast, the amax and the transposed copy are one pass over
// 128x128 tiles (the cast kernel with a LayerNorm element operation, in
// cast.cu), after a pass that computes the per-row statistics.
#include <cuda_bf16.h>

#include "common.cuh"

namespace fp8dl {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf16r(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// ---------------------------------------------------------------------------
// Row statistics of LayerNorm: warp per row, the row held in registers,
//   mu = sum(x)/C, var = sum((x-mu)^2)/C (two passes over the registers), rs = 1/sqrt(var+eps).
// ---------------------------------------------------------------------------
template <int CPL>
__global__ void __launch_bounds__(256) ln_stats_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                       float eps, float *__restrict__ mu_out,
                                                       float *__restrict__ rs_out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t nchunks = cols / 8;
    const float inv_cols = 1.0f / (float)cols;
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const uint16_t *xr = x + r * cols;
        uint4 v[CPL];
#pragma unroll
        for (int i = 0; i < CPL; i++)
            if (lane + 32 * i < nchunks) v[i] = ldg_stream(xr + 8 * (lane + 32 * i));
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < CPL; i++)
            if (lane + 32 * i < nchunks) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int q = 0; q < 4; q++) s += bf16_lo(w[q]) + bf16_hi(w[q]);
            }
        const float mean = warp_sum(s) * inv_cols;
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < CPL; i++)
            if (lane + 32 * i < nchunks) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float a = bf16_lo(w[q]) - mean, b = bf16_hi(w[q]) - mean;
                    ss += a * a + b * b;
                }
            }
        const float var = warp_sum(ss) * inv_cols;
        if (lane == 0) {
            mu_out[r] = mean;
            rs_out[r] = 1.0f / sqrtf(var + eps);
        }
    }
}

fp8dl_status launch_layernorm_tile_cast(const void *x, const float *mu, const float *rs, const void *gamma,
                                        const void *beta, int64_t rows, int64_t cols, int fmt, const float *scale,
                                        uint8_t *out, uint8_t *out_t, float *amax, void *y, int sms,
                                        cudaStream_t st);

// ---------------------------------------------------------------------------
// LayerNorm backward, given the forward's per-row mu and rs:
//   xhat = (x - mu) * rs, g = dy * gamma
//   dx = rs * (g - mean(g) - xhat * mean(g * xhat))          (bf16 out)
//   dgamma = sum_rows dy * xhat, dbeta = sum_rows dy           (fp32 out)
// Pass 1 (warp per row): the two row means.  Pass 2 (128 x 128 tiles): dx and
// per-tile column partials of dgamma/dbeta; pass 3 sums the partials in order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) ln_bwd_rowsum_kernel(const uint16_t *__restrict__ dy,
                                                            const uint16_t *__restrict__ x,
                                                            const uint16_t *__restrict__ gamma,
                                                            const float *__restrict__ mu,
                                                            const float *__restrict__ rs, int64_t rows, int64_t cols,
                                                            float *__restrict__ c12) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const float inv_cols = 1.0f / (float)cols;
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float m = mu[r], s = rs[r];
        float s1 = 0.0f, s2 = 0.0f;
        for (int64_t c = lane; c < cols / 8; c += 32) {
            const uint4 dv = ldg_stream(dy + r * cols + 8 * c);
            const uint4 xv = ldg_stream(x + r * cols + 8 * c);
            const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(gamma + 8 * c));
            const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w},
                           gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float g0 = bf16_lo(dw[q]) * bf16_lo(gw[q]), g1 = bf16_hi(dw[q]) * bf16_hi(gw[q]);
                const float h0 = (bf16_lo(xw[q]) - m) * s, h1 = (bf16_hi(xw[q]) - m) * s;
                s1 += g0 + g1;
                s2 += g0 * h0 + g1 * h1;
            }
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        if (lane == 0) {
            c12[2 * r] = s1 * inv_cols;
            c12[2 * r + 1] = s2 * inv_cols;
        }
    }
}

constexpr int LB_ROWS = 128, LB_COLS = 128;

__global__ void __launch_bounds__(256) ln_bwd_tile_kernel(const uint16_t *__restrict__ dy,
                                                          const uint16_t *__restrict__ x,
                                                          const uint16_t *__restrict__ gamma,
                                                          const float *__restrict__ mu, const float *__restrict__ rs,
                                                          const float *__restrict__ c12, int64_t rows, int64_t cols,
                                                          uint16_t *__restrict__ dx, float *__restrict__ part) {
    __shared__ __align__(16) float red_g[8][LB_COLS];
    __shared__ __align__(16) float red_b[8][LB_COLS];
    const int t = threadIdx.x, cb = t & 7, rb = t >> 3, lane = t & 31, wi = t >> 5;
    const int64_t tiles_c = (cols + LB_COLS - 1) / LB_COLS;
    const int64_t tiles = ((rows + LB_ROWS - 1) / LB_ROWS) * tiles_c;
    const int64_t n_rt = (rows + LB_ROWS - 1) / LB_ROWS;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t r0 = (tile / tiles_c) * LB_ROWS, c0 = (tile % tiles_c) * LB_COLS;
        float pg[16], pb[16];
#pragma unroll
        for (int j = 0; j < 16; j++) pg[j] = pb[j] = 0.0f;
        if (r0 + 4 * rb < rows && c0 + 16 * cb < cols) {
            const int64_t col = c0 + 16 * cb;
            const uint4 g0 = __ldg(reinterpret_cast<const uint4 *>(gamma + col));
            const uint4 g1 = __ldg(reinterpret_cast<const uint4 *>(gamma + col + 8));
            const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int64_t r = r0 + 4 * rb + i;
                const float m = mu[r], s = rs[r], c1 = c12[2 * r], c2 = c12[2 * r + 1];
                const uint4 d0 = ldg_stream(dy + r * cols + col), d1 = ldg_stream(dy + r * cols + col + 8);
                const uint4 x0 = ldg_stream(x + r * cols + col), x1 = ldg_stream(x + r * cols + col + 8);
                const uint32_t dw[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                uint32_t ow[8];
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const float d_lo = bf16_lo(dw[q]), d_hi = bf16_hi(dw[q]);
                    const float h_lo = (bf16_lo(xw[q]) - m) * s, h_hi = (bf16_hi(xw[q]) - m) * s;
                    const float o_lo = s * (d_lo * bf16_lo(gw[q]) - c1 - h_lo * c2);
                    const float o_hi = s * (d_hi * bf16_hi(gw[q]) - c1 - h_hi * c2);
                    pg[2 * q] += d_lo * h_lo;
                    pg[2 * q + 1] += d_hi * h_hi;
                    pb[2 * q] += d_lo;
                    pb[2 * q + 1] += d_hi;
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(o_lo, o_hi);
                    ow[q] = *reinterpret_cast<uint32_t *>(&b2);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(dx + r * cols + col);
                dst[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                dst[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
            }
        }
#pragma unroll
        for (int j = 0; j < 16; j++) {
            pg[j] += __shfl_xor_sync(0xffffffffu, pg[j], 8);
            pg[j] += __shfl_xor_sync(0xffffffffu, pg[j], 16);
            pb[j] += __shfl_xor_sync(0xffffffffu, pb[j], 8);
            pb[j] += __shfl_xor_sync(0xffffffffu, pb[j], 16);
        }
        if (lane < 8) {
            float4 *dg4 = reinterpret_cast<float4 *>(&red_g[wi][16 * cb]);
            float4 *db4 = reinterpret_cast<float4 *>(&red_b[wi][16 * cb]);
#pragma unroll
            for (int j = 0; j < 4; j++) {
                dg4[j] = make_float4(pg[4 * j], pg[4 * j + 1], pg[4 * j + 2], pg[4 * j + 3]);
                db4[j] = make_float4(pb[4 * j], pb[4 * j + 1], pb[4 * j + 2], pb[4 * j + 3]);
            }
        }
        __syncthreads();
        if (t < LB_COLS && c0 + t < cols) {
            float sg = 0.0f, sb = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; k++) {
                sg += red_g[k][t];
                sb += red_b[k][t];
            }
            const int64_t tr = r0 / LB_ROWS;
            part[tr * cols + c0 + t] = sg;
            part[(n_rt + tr) * cols + c0 + t] = sb;
        }
        __syncthreads();
    }
}

// dgamma/dbeta[c] = sum over row tiles of the partials, fixed order (see colsum_reduce_kernel).
__global__ void __launch_bounds__(256) ln_bwd_reduce_kernel(const float *__restrict__ part, int64_t n_rt, int64_t cols,
                                                            float *__restrict__ dgamma, float *__restrict__ dbeta) {
    __shared__ float pg[8][32], pb[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t c = blockIdx.x * (int64_t)32 + lane;
    float sg = 0.0f, sb = 0.0f;
    if (c < cols)
        for (int64_t k = w; k < n_rt; k += 8) {
            sg += part[k * cols + c];
            sb += part[(n_rt + k) * cols + c];
        }
    pg[w][lane] = sg;
    pb[w][lane] = sb;
    __syncthreads();
    if (w == 0 && c < cols) {
        float a = 0.0f, b = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            a += pg[k][lane];
            b += pb[k][lane];
        }
        dgamma[c] = a;
        dbeta[c] = b;
    }
}

}  // namespace fp8dl

using namespace fp8dl;

extern "C" {

fp8dl_status fp8_layernorm_cast(const void *x, int64_t rows, int64_t cols, const void *gamma, const void *beta,
                                float eps, int32_t out_dtype, const float *scale, uint8_t *out, uint8_t *out_t,
                                float *amax, float *mu, float *rsigma, void *y, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_layernorm_cast");
    FP8DL_CHECK_ARG(x && gamma && beta && mu && rsigma, "x, gamma, beta, mu and rsigma must be non-NULL");
    FP8DL_CHECK_ARG(out_dtype == FP8DL_E4M3 || out_dtype == FP8DL_E5M2, "out_dtype must be E4M3 or E5M2");
    FP8DL_CHECK_ARG(!(out || out_t) || scale != nullptr, "scale is NULL but an FP8 output was requested");
    FP8DL_CHECK_ARG(eps >= 0.0f, "eps must be >= 0");
    if (!dim_ok(rows, 16) || !dim_ok(cols, 16) || cols > 8192)
        return fail(FP8DL_ERR_SHAPE, "rows (%lld) and cols (%lld) must be positive multiples of 16, cols <= 8192",
                    (long long)rows, (long long)cols);
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out) || !aligned16(out_t) ||
        !aligned16(y))
        return fail(FP8DL_ERR_ALIGN, "x, gamma, beta, out, out_t and y must be 16-byte aligned");
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    cudaStream_t st = (cudaStream_t)stream;
    // pass 1: per-row statistics (one read of x); pass 2: normalise + cast in 128x128 tiles
    const int64_t chunks_per_lane = (cols / 8 + 31) / 32;
    const int64_t row_ctas = (rows + 7) / 8;
    const unsigned g1 = (unsigned)(row_ctas < (int64_t)sms * 8 ? row_ctas : (int64_t)sms * 8);
    auto X = static_cast<const uint16_t *>(x);
    if (chunks_per_lane <= 4)
        ln_stats_kernel<4><<<g1, 256, 0, st>>>(X, rows, cols, eps, mu, rsigma);
    else if (chunks_per_lane <= 8)
        ln_stats_kernel<8><<<g1, 256, 0, st>>>(X, rows, cols, eps, mu, rsigma);
    else if (chunks_per_lane <= 16)
        ln_stats_kernel<16><<<g1, 256, 0, st>>>(X, rows, cols, eps, mu, rsigma);
    else
        ln_stats_kernel<32><<<g1, 256, 0, st>>>(X, rows, cols, eps, mu, rsigma);
    FP8DL_TRY(check_launch("fp8_layernorm_cast(statistics)"));
    if (!(out || out_t || amax || y)) return FP8DL_OK;
    return launch_layernorm_tile_cast(x, mu, rsigma, gamma, beta, rows, cols, out_dtype, scale, out, out_t, amax, y,
                                      sms, st);
}

size_t fp8_layernorm_bwd_workspace_size(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    const size_t n_rt = (size_t)((rows + LB_ROWS - 1) / LB_ROWS);
    return (2 * (size_t)rows + 2 * n_rt * (size_t)cols) * sizeof(float);
}

fp8dl_status fp8_layernorm_bwd(const void *dy, const void *x, const void *gamma, const float *mu,
                               const float *rsigma, int64_t rows, int64_t cols, void *dx, float *dgamma,
                               float *dbeta, void *workspace, size_t workspace_bytes, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_layernorm_bwd");
    FP8DL_CHECK_ARG(dy && x && gamma && mu && rsigma && dx && dgamma && dbeta,
                    "dy, x, gamma, mu, rsigma, dx, dgamma and dbeta must be non-NULL");
    if (!dim_ok(rows, 16) || !dim_ok(cols, 16))
        return fail(FP8DL_ERR_SHAPE, "rows (%lld) and cols (%lld) must be positive multiples of 16", (long long)rows,
                    (long long)cols);
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(dx) || !aligned16(workspace))
        return fail(FP8DL_ERR_ALIGN, "dy, x, gamma, dx and workspace must be 16-byte aligned");
    if (!workspace || workspace_bytes < fp8_layernorm_bwd_workspace_size(rows, cols))
        return fail(FP8DL_ERR_WORKSPACE, "fp8_layernorm_bwd needs a workspace of %zu bytes",
                    fp8_layernorm_bwd_workspace_size(rows, cols));
    int sms = 0;
    FP8DL_TRY(current_device(nullptr, &sms));
    cudaStream_t st = (cudaStream_t)stream;
    float *c12 = static_cast<float *>(workspace);
    float *part = c12 + 2 * rows;
    auto DY = static_cast<const uint16_t *>(dy);
    auto X = static_cast<const uint16_t *>(x);
    auto G = static_cast<const uint16_t *>(gamma);
    const int64_t row_ctas = (rows + 7) / 8;
    ln_bwd_rowsum_kernel<<<(unsigned)(row_ctas < (int64_t)sms * 8 ? row_ctas : (int64_t)sms * 8), 256, 0, st>>>(
        DY, X, G, mu, rsigma, rows, cols, c12);
    FP8DL_TRY(check_launch("fp8_layernorm_bwd(row sums)"));
    const int64_t n_rt = (rows + LB_ROWS - 1) / LB_ROWS;
    const int64_t tiles = n_rt * ((cols + LB_COLS - 1) / LB_COLS);
    ln_bwd_tile_kernel<<<(unsigned)(tiles < (int64_t)sms * 4 ? tiles : (int64_t)sms * 4), 256, 0, st>>>(
        DY, X, G, mu, rsigma, c12, rows, cols, static_cast<uint16_t *>(dx), part);
    FP8DL_TRY(check_launch("fp8_layernorm_bwd(dx)"));
    ln_bwd_reduce_kernel<<<(unsigned)((cols + 31) / 32), 256, 0, st>>>(part, n_rt, cols, dgamma, dbeta);
    return check_launch("fp8_layernorm_bwd(reduce)");
}

}  // extern "C"
