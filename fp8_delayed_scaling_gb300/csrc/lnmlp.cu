// lnmlp.cu — LayerNorm pieces of the LayerNormMLP path: LayerNorm forward fused
// with the FP8 cast of its output, and the LayerNorm backward.
//
// "NVIDIA Transformer Engine 加速训练教程" builds blocks from te.LayerNormMLP
// (LayerNorm -> fc1 -> GELU -> fc2) and mirrors them in plain PyTorch with
// nn.LayerNorm (biased variance).  Under delayed scaling ("FP8 低精度训练：
// Transformer Engine 简析" §三.1/§三.3) the LayerNorm output is what fc1 casts,
// and its scale is known before the LayerNorm runs, so normalisation, bf16
// rounding, the FP8 cast, the amax and the transposed copy happen in the pass
// that reads x.
//
// Two implementations of each direction:
//  - cluster path (cols a multiple of 512, at most 16 x 512): a thread-block
//    cluster owns blocks of rows (32 forward, 16 backward); CTA k of the cluster
//    stages columns [512k, 512k + 512) of the block in shared memory, the CTAs
//    push their per-row partial sums into each other's shared memory, and x
//    (and dy) are read from HBM once;
//  - tile path (any other width): a warp-per-row statistics pass, then 128 x 128
//    tiles (the cast kernel with a LayerNorm element operation, in cast.cu).
#include <cuda_bf16.h>
#include <stdlib.h>

#include "common.cuh"
#include "tc.cuh"

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
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
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
                                        cudaStream_t st, bool pdl);

// ---------------------------------------------------------------------------
// Cluster path.  CTA `rank` of a cluster covers columns [LC_COLS*rank,
// LC_COLS*rank + LC_COLS) of every row block the cluster owns; the cluster's
// blocks are cid, cid + n_clusters, ... (block j of the cluster below).  The
// block is staged in shared memory with cp.async (three buffers).
//
// Software pipeline, per CTA, in iteration j:
//   - block j+2 is copied into shared memory;
//   - the row partials of block j+1 are reduced over the CTA and pushed with
//     st.async into exchange slot (j+1) mod 4 of every CTA of the cluster
//     (this CTA's entry of each), completing on that CTA's slot barrier;
//   - the CTA waits on its own slot barrier for block j (pushed one iteration
//     earlier), merges the CTAs' partials, re-arms the barrier for block j+4,
//     and block j is normalised and written.
// The forward reduces block j+1 and then gathers block j, spreading the merge
// over all threads (one barrier publishes both); the backward, with shorter
// blocks, pushes block j+1 (warp 0) before block j is gathered (warp 1), so
// that block j's pushes have longer to arrive.
// The exchange's latency is thus hidden behind a whole block's work, and no
// cluster-wide barrier or release fence (which would also wait for the
// previous block's global stores) sits in the loop.  Slots rotate over four
// blocks: a CTA pushes block j+4 only after it has received block j+2 from
// every CTA, and each CTA pushes block j+2 after it has read block j.
// A barrier at the top of every iteration separates the refill of a buffer
// from the previous block's reads of it.
// ---------------------------------------------------------------------------
constexpr int LC_COLS = 512, LC_THREADS = 256, LC_WARPS = LC_THREADS / 32, LC_MAX_CLUSTER = 16, LC_NBUF = 3;
constexpr int LC_SLOTS = 4;  // exchange slots, by block number modulo 4
constexpr int LF_ROWS = 32;  // forward block: two halves of 16 rows, 32-byte column segments of out_t
constexpr int LB_BLK = 16;   // backward block: 4 rows per thread
constexpr int LB_CTAS = 2;   // backward CTAs per SM (registers and shared memory sized for it)
constexpr int LF_BUF = LF_ROWS * LC_COLS * 2;      // one staged x block
constexpr int LF_SMEM = LC_NBUF * LF_BUF;  // then LC_SLOTS x cluster size x LF_ROWS pushed float2
// dynamic shared memory of a launch: staged blocks plus `slot_rows` rows of pushed partials per
// slot and CTA of the cluster
constexpr int ln_smem(int base, int slot_rows, int cl) { return base + LC_SLOTS * cl * slot_rows * 8; }
constexpr int LB_SMEM = LC_NBUF * 2 * LB_BLK * LC_COLS * 2;  // three staged (dy, x) blocks

__device__ __forceinline__ int next_buf(int b) { return b == LC_NBUF - 1 ? 0 : b + 1; }

// rows 0..3 x columns 0..3 of bytes (w[k] = row k, column j in byte j) -> column j's 4 rows in col[j].
__device__ __forceinline__ void transpose4x4_bytes(const uint32_t (&w)[4], uint32_t (&col)[4]) {
    const uint32_t t0 = __byte_perm(w[0], w[1], 0x5140), t1 = __byte_perm(w[2], w[3], 0x5140);
    const uint32_t t2 = __byte_perm(w[0], w[1], 0x7362), t3 = __byte_perm(w[2], w[3], 0x7362);
    col[0] = __byte_perm(t0, t1, 0x5410);
    col[1] = __byte_perm(t0, t1, 0x7632);
    col[2] = __byte_perm(t2, t3, 0x5410);
    col[3] = __byte_perm(t2, t3, 0x7632);
}

// Asynchronous global -> shared copies (the issuing thread waits for its own groups).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A bf16x2 word as two floats (low half first), and two floats rounded to a bf16x2 word.
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_bf16x2(float2 v) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ float2 shfl_xor2(float2 v, int o) {
    return make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
}

// Mean and sum of squared deviations of two groups of n values each, combined
// (Chan, Golub and LeVeque's pairwise update with equal counts:
// M2 = M2_a + M2_b + (m_a - m_b)^2 * n / 2).  Symmetric in a and b.
__device__ __forceinline__ float2 chan_equal(float2 a, float2 b, float half_n) {
    const float d = a.x - b.x;
    return make_float2((a.x + b.x) * 0.5f, (a.y + b.y) + d * d * half_n);
}

// LayerNorm forward + cast.  Warp w covers columns 64w .. 64w+63 of the CTA's
// slab; lane (rg = lane >> 2, cg = lane & 3) holds columns 64w + 16cg .. +15 of
// rows 4rg .. 4rg+3 of the 32-row block.  In shared memory the 16-byte chunk
// ch of row r sits at chunk ch ^ ((r >> 2) & 7) of its row, so the two chunk
// loads of a lane's row hit every bank group four times per warp.
// Statistics: each lane takes the mean and M2 of its 16 values of a row (two
// passes over registers); the four lanes of a row group and then the eight
// warps merge them (Chan's equal-count update), and the cluster's slabs are
// combined as mean = sum_k m_k / n_slabs, M2 = sum_k (M2_k + 512 (m_k - mean)^2)
// (each sum a fixed butterfly over the slabs); var = M2 / cols,
// rs = 1/sqrt(var + eps).  Every CTA then normalises its slab:
// y = bf16((x - mu) * rs * gamma + beta), codes = cvt(y * scale), written
// row-major (out: 16 bytes per lane and row) and transposed (out_t: the four
// rows of a column are one 4-byte word, and the eight row groups of a warp
// fill one 32-byte segment).
template <int FMT>
__global__ void __launch_bounds__(LC_THREADS, 2) ln_fwd_cluster_kernel(
    const uint16_t *__restrict__ x, const uint16_t *__restrict__ gamma, const uint16_t *__restrict__ beta,
    int64_t rows, int64_t cols, float eps, const float *__restrict__ scale_p, uint8_t *__restrict__ out,
    uint8_t *__restrict__ out_t, float *__restrict__ amax_p, float *__restrict__ mu_out, float *__restrict__ rs_out,
    uint16_t *__restrict__ y) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    extern __shared__ __align__(128) uint8_t lsm[];      // [LC_NBUF][LF_ROWS][LC_COLS] bf16, then the slots
    __shared__ float2 wst[LC_WARPS][LF_ROWS + 1];        // per-warp (mean, M2) of 64 values of a row
    __shared__ __align__(8) uint64_t xbar[LC_SLOTS];     // slot s complete: every CTA's slabs of its block arrived
    __shared__ float2 stat[LF_ROWS];                     // mean, rsigma
    __shared__ float wmax[LC_WARPS];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int rg = lane >> 2, cg = lane & 3;
    const int c0 = 8 * w + 2 * cg;  // the lane's first 16-byte chunk of a row (of 64)
    const uint32_t rank = cluster_ctarank(), ncta = cluster_nctarank();
    const int64_t col0 = (int64_t)rank * LC_COLS, col = col0 + 8 * c0;
    const int64_t nblk = (rows + LF_ROWS - 1) / LF_ROWS;
    const int64_t cid = blockIdx.x / ncta, ncl = gridDim.x / ncta;
    const int64_t nb = cid < nblk ? (nblk - cid + ncl - 1) / ncl : 0;  // this cluster's blocks
    float2 *gath = reinterpret_cast<float2 *>(lsm + LF_SMEM);  // [LC_SLOTS][ncta][LF_ROWS], pushed by the CTAs
    const uint32_t push_bytes = ncta * LF_ROWS * (uint32_t)sizeof(float2);  // per slot and block
    const float scale = (out || out_t) ? __ldg(scale_p) : 1.0f;
    const float2 sc2 = make_float2(scale, scale);
    uint8_t *const out_tb = out_t ? out_t + col * rows + 4 * rg : nullptr;  // plus r0: the lane's first out_t word
    float2 g2[8], b2[8];
    {
        const uint4 ga = __ldg(reinterpret_cast<const uint4 *>(gamma + col));
        const uint4 gb = __ldg(reinterpret_cast<const uint4 *>(gamma + col + 8));
        const uint4 ba = __ldg(reinterpret_cast<const uint4 *>(beta + col));
        const uint4 bb = __ldg(reinterpret_cast<const uint4 *>(beta + col + 8));
        const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
        const uint32_t bw[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
#pragma unroll
        for (int q = 0; q < 8; q++) {
            g2[q] = bf16x2_f2(gw[q]);
            b2[q] = bf16x2_f2(bw[q]);
        }
    }
    // Copy block j into buffer `buf`: 32 rows x 64 chunks of 16 bytes, 8 per thread (rows
    // t/64 + 4i, chunk t % 64), a warp per half row; chunk ch of row r goes to chunk
    // ch ^ ((r >> 2) & 7), which is ch ^ i here.
    const int crow = t >> 6, cch = t & 63;
    const uint16_t *xsrc = x + (int64_t)crow * cols + col0 + 8 * cch;
    const uint32_t sdst = smem_u32(lsm) + (crow * LC_COLS) * 2;
    auto issue = [&](int64_t j, int buf) {
        if (j < nb) {
            const int64_t r0 = (cid + j * ncl) * LF_ROWS;
            const uint16_t *src = xsrc + r0 * cols;
            const int64_t lim = rows - r0 - crow;  // copy i is valid while 4i < lim
            const uint32_t dst = sdst + buf * LF_BUF;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const bool valid = 4 * i < lim;
                cp_async16(dst + i * 4 * LC_COLS * 2 + 16 * (cch ^ i), valid ? src + 4 * i * cols : x, valid);
            }
        }
        cp_async_commit();  // possibly empty: one group per block keeps the wait counts uniform
    };
    // the lane's 16 values of row 4rg + i, as eight bf16x2 words
    const uint8_t *xl0 = lsm + 4 * rg * LC_COLS * 2 + 16 * (c0 ^ rg), *xl1 = lsm + 4 * rg * LC_COLS * 2 + 16 * ((c0 + 1) ^ rg);
    auto xrow = [&](int buf, int i, uint32_t (&v)[8]) {
        const uint4 a = *reinterpret_cast<const uint4 *>(xl0 + buf * LF_BUF + i * LC_COLS * 2);
        const uint4 b = *reinterpret_cast<const uint4 *>(xl1 + buf * LF_BUF + i * LC_COLS * 2);
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
    };
    // Per-warp (mean, M2) of the staged block in `buf`, into wst.
    auto partials = [&](int buf) {
        float2 s[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t q[8];
            xrow(buf, i, q);
            float2 v[8];
#pragma unroll
            for (int k = 0; k < 8; k++) v[k] = bf16x2_f2(q[k]);
            const float2 s01 = __fadd2_rn(__fadd2_rn(v[0], v[1]), __fadd2_rn(v[2], v[3]));
            const float2 s23 = __fadd2_rn(__fadd2_rn(v[4], v[5]), __fadd2_rn(v[6], v[7]));
            const float2 sum = __fadd2_rn(s01, s23);
            const float m = (sum.x + sum.y) * 0.0625f;
            const float2 nm = make_float2(-m, -m);
            float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const float2 d = __fadd2_rn(v[k], nm);
                acc = __ffma2_rn(d, d, acc);
            }
            s[i] = make_float2(m, acc.x + acc.y);
        }
        // reduce-scatter over the four lanes of the row group: lane bit 0, then bit 1
        const bool u1 = lane & 1, u2 = lane & 2;
        float2 k2[2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const float2 send = u1 ? s[i] : s[i + 2], keep = u1 ? s[i + 2] : s[i];
            k2[i] = chan_equal(keep, shfl_xor2(send, 1), 8.0f);
        }
        const float2 send = u2 ? k2[0] : k2[1], keep = u2 ? k2[1] : k2[0];
        wst[w][4 * rg + 2 * u1 + u2] = chan_equal(keep, shfl_xor2(send, 2), 16.0f);
    };
    // The exchange is spread over all threads: thread t serves row gr = t / 8 of the block and
    // the slabs (warps, then cluster ranks) gk = t % 8 and gk + 8; the eight threads of a row
    // merge by butterfly, which leaves the same bits in each of them.
    const int gr = t >> 3, gk = t & 7;
    // After a barrier: the CTA's (mean, M2) of row gr, merged over the eight warps, pushed into
    // slot `slot` of every CTA of the cluster (this CTA's entry), completing on that CTA's barrier.
    auto push = [&](int slot) {
        float2 v = wst[gk][gr];
        v = chan_equal(v, shfl_xor2(v, 1), 32.0f);
        v = chan_equal(v, shfl_xor2(v, 2), 64.0f);
        v = chan_equal(v, shfl_xor2(v, 4), 128.0f);
        const uint32_t la = smem_u32(&gath[(slot * ncta + rank) * LF_ROWS + gr]), lb = smem_u32(&xbar[slot]);
        for (uint32_t k = gk; k < ncta; k += 8) st_async_f2(mapa_shared(la, k), v, mapa_shared(lb, k));
    };
    // Statistics of block j (row gr) from every CTA's slab in slot `slot`: mean = sum_k m_k / ncta,
    // M2 = sum_k (M2_k + LC_COLS (m_k - mean)^2).  A wait that runs out leaves NaN statistics.
    auto gather = [&](int64_t j, int slot) {
        const bool arrived = mbar_wait_bounded(smem_u32(&xbar[slot]), (uint32_t)((j / LC_SLOTS) & 1));
        const bool ha = gk < (int)ncta, hb = gk + 8 < (int)ncta;
        const float2 pa = ha ? gath[(slot * ncta + gk) * LF_ROWS + gr] : make_float2(0.0f, 0.0f);
        const float2 pb = hb ? gath[(slot * ncta + gk + 8) * LF_ROWS + gr] : make_float2(0.0f, 0.0f);
        float sm = arrived ? pa.x + pb.x : __int_as_float(0x7fc00000);
        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
        sm += __shfl_xor_sync(0xffffffffu, sm, 4);
        const float mean = sm / (float)ncta;
        const float da = pa.x - mean, db = pb.x - mean;
        float m2 = (ha ? pa.y + da * da * (float)LC_COLS : 0.0f) + (hb ? pb.y + db * db * (float)LC_COLS : 0.0f);
        m2 += __shfl_xor_sync(0xffffffffu, m2, 1);
        m2 += __shfl_xor_sync(0xffffffffu, m2, 2);
        m2 += __shfl_xor_sync(0xffffffffu, m2, 4);
        if (gk == 0) {
            const int64_t r0 = (cid + j * ncl) * LF_ROWS;
            const float rsig = 1.0f / sqrtf(m2 / (float)cols + eps);
            stat[gr] = make_float2(mean, rsig);
            if (rank == 0 && r0 + gr < rows) {
                mu_out[r0 + gr] = mean;
                rs_out[r0 + gr] = rsig;
            }
        }
        // the slot's next block: its barrier counts the pushes of block j + LC_SLOTS
        if (t == 0 && j + LC_SLOTS < nb) mbar_expect_tx(smem_u32(&xbar[slot]), push_bytes);
    };
    if (t == 0) {
        for (int k = 0; k < LC_SLOTS; k++) mbar_init(smem_u32(&xbar[k]), 1);
        mbar_fence_init();
    }
    cluster_sync();  // every CTA's barriers are initialised before anything is pushed to them
    if (t == 0)
        for (int k = 0; k < LC_SLOTS && k < nb; k++) mbar_expect_tx(smem_u32(&xbar[k]), push_bytes);
    uint32_t amax2 = 0;  // bf16x2 running |y| maxima
    if (nb > 0) {  // always, as no more clusters than blocks are launched
        issue(0, 0);
        issue(1, 1);
        cp_async_wait<1>();
        __syncthreads();  // block 0 was copied by every thread
        partials(0);
        __syncthreads();
        push(0);
    }
    int buf = 0, slot = 0;
    for (int64_t j = 0; j < nb; j++) {
        const int64_t r0 = (cid + j * ncl) * LF_ROWS;
        const int nslot = (slot + 1) & (LC_SLOTS - 1);
        cp_async_wait<0>();  // this thread's copies of block j+1 have landed (the only group in flight)
        __syncthreads();     // ... everyone's; and every thread is past block j-1, whose buffer is refilled now
        issue(j + 2, next_buf(next_buf(buf)));
        // every warp reduces block j+1, then gathers block j (pushed during the previous
        // iteration); one barrier publishes both, then block j+1 is pushed
        if (j + 1 < nb) partials(next_buf(buf));
        gather(j, slot);
        __syncthreads();
        if (j + 1 < nb) push(nslot);
        if (r0 + 4 * rg < rows) {  // rows are a multiple of 16: a row group is all in or all out
            const int64_t rowoff = (r0 + 4 * rg) * cols + col;  // of this lane's first element
            uint32_t codes[4][4];  // [row][column quad]
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float2 sr = stat[4 * rg + i];
                const float2 nmu = make_float2(-sr.x, -sr.x), rs2 = make_float2(sr.y, sr.y);
                uint32_t q[8], yw[8];
                xrow(buf, i, q);
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    // y = bf16((x - mu) * rs * gamma + beta), two at a time
                    yw[k] = f2_bf16x2(__ffma2_rn(__fmul2_rn(__fadd2_rn(bf16x2_f2(q[k]), nmu), rs2), g2[k], b2[k]));
                    amax2 = bf16x2_absmax(amax2, yw[k]);
                }
                if (y) {
                    uint4 *yp = reinterpret_cast<uint4 *>(y + rowoff + i * cols);
                    yp[0] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
                    yp[1] = make_uint4(yw[4], yw[5], yw[6], yw[7]);
                }
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const float2 ya = __fmul2_rn(bf16x2_f2(yw[2 * k]), sc2), yb = __fmul2_rn(bf16x2_f2(yw[2 * k + 1]), sc2);
                    codes[i][k] = pack4<FMT>(ya.x, ya.y, yb.x, yb.y);
                }
                if (out)
                    *reinterpret_cast<uint4 *>(out + rowoff + i * cols) =
                        make_uint4(codes[i][0], codes[i][1], codes[i][2], codes[i][3]);
            }
            if (out_t) {
                uint8_t *ot = out_tb + r0;  // column `col`, row r0 + 4rg
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const uint32_t wr[4] = {codes[0][k], codes[1][k], codes[2][k], codes[3][k]};
                    uint32_t cw[4];  // cw[jj]: rows 4rg .. 4rg+3 of column 4k + jj
                    transpose4x4_bytes(wr, cw);
#pragma unroll
                    for (int jj = 0; jj < 4; jj++) {
                        *reinterpret_cast<uint32_t *>(ot) = cw[jj];
                        ot += rows;
                    }
                }
            }
        }
        buf = next_buf(buf);
        slot = nslot;
    }
    cp_async_wait<0>();
    if (amax_p) {
        const float m = warp_max(fmaxf(fabsf(bf16_lo(amax2)), fabsf(bf16_hi(amax2))));
        if (lane == 0) wmax[w] = m;
        __syncthreads();
        if (t == 0) {
            float mm = wmax[0];
            for (int k = 1; k < LC_WARPS; k++) mm = fmaxf(mm, wmax[k]);
            atomic_max_nonneg(amax_p, mm);
        }
    }
    cluster_sync();  // every push to this CTA has arrived (it waited for them); none leaves before the rest
}

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
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
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
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
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
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
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

// Sum of the float2 partials of R rows (R = 2 or 4) over a warp, scattered:
// lane l returns the row given by its top bits (R = 4: 2*b4 + b3; R = 2: b4).
template <int R>
__device__ __forceinline__ float2 warp_sum_rows(const float2 (&s)[R], int lane) {
    static_assert(R == 2 || R == 4, "2 or 4 rows");
    float2 r;
    if constexpr (R == 4) {
        const bool u4 = lane & 16, u3 = lane & 8;
        float2 k2[2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const float2 send = u4 ? s[i] : s[i + 2], keep = u4 ? s[i + 2] : s[i];
            const float2 p = shfl_xor2(send, 16);
            k2[i] = make_float2(keep.x + p.x, keep.y + p.y);
        }
        const float2 send = u3 ? k2[0] : k2[1], keep = u3 ? k2[1] : k2[0];
        const float2 p = shfl_xor2(send, 8);
        r = make_float2(keep.x + p.x, keep.y + p.y);
    } else {
        const bool u4 = lane & 16;
        const float2 send = u4 ? s[0] : s[1], keep = u4 ? s[1] : s[0];
        const float2 p = shfl_xor2(send, 16);
        r = make_float2(keep.x + p.x, keep.y + p.y);
#pragma unroll
        for (int o = 8; o > 4; o >>= 1) {
            const float2 q = shfl_xor2(r, o);
            r = make_float2(r.x + q.x, r.y + q.y);
        }
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
        const float2 q = shfl_xor2(r, o);
        r = make_float2(r.x + q.x, r.y + q.y);
    }
    return r;
}

// LayerNorm backward on the cluster layout, with the forward's pipeline.  Per
// row block of BLK rows, thread t holds the 8 columns starting at
// LC_COLS*rank + 8*(t & 63) of rows (BLK/4)*(t >> 6) .. +BLK/4-1 and copies and
// reads only its own 16-byte chunks of dy and x.  Each thread forms
// g = dy * gamma and xhat = (x - mu) * rs for its slab; the row partials of
// sum(g) and sum(g * xhat) are published for the cluster (one block ahead),
// summed over the CTAs in rank order, and
//   dx = rs * (g - c1 - xhat * c2) = (x - mu) * k2 + (rs * g + k1),
//   c1 = mean(g), c2 = mean(g * xhat), k1 = -rs * c1, k2 = -rs^2 * c2,
// is written from the staged block.  Each thread keeps the column partials of dgamma (dy * xhat) and dbeta
// (dy) of its 8 columns across all of the cluster's blocks; at the end the CTA
// writes one partial row per cluster, part[cluster][col] (dgamma) and
// part[n_clusters + cluster][col] (dbeta), which ln_bwd_reduce_kernel sums in
// cluster order.
template <int BLK>
__global__ void __launch_bounds__(LC_THREADS, LB_CTAS) ln_bwd_cluster_kernel(
    const uint16_t *__restrict__ dy, const uint16_t *__restrict__ x, const uint16_t *__restrict__ gamma,
    const float *__restrict__ mu, const float *__restrict__ rs, int64_t rows, int64_t cols,
    uint16_t *__restrict__ dx, float *__restrict__ part) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    constexpr int RPT = BLK / 4;                     // rows per thread
    constexpr int BUF = 2 * BLK * LC_COLS * 2;       // one staged (dy, x) block
    extern __shared__ __align__(128) uint8_t lsm[];  // [LC_NBUF][dy, x][BLK][LC_COLS] bf16, then the slots
    __shared__ float2 wsum[LC_WARPS][RPT];
    __shared__ __align__(8) uint64_t xbar[LC_SLOTS];  // slot s complete: every CTA's partials of its block arrived
    __shared__ float2 cst[BLK];                      // mean(g), mean(g * xhat)
    __shared__ float mrs[LC_NBUF][2][BLK];           // [buffer][mu, rs][row]
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int c = t & 63, g = t >> 6;
    const uint32_t rank = cluster_ctarank(), ncta = cluster_nctarank();
    const int64_t col0 = (int64_t)rank * LC_COLS, col = col0 + 8 * c;
    const int64_t nblk = (rows + BLK - 1) / BLK;
    const int64_t cid = blockIdx.x / ncta, ncl = gridDim.x / ncta;
    const int64_t nb = cid < nblk ? (nblk - cid + ncl - 1) / ncl : 0;
    float2 *gath = reinterpret_cast<float2 *>(lsm + LC_NBUF * BUF);  // [LC_SLOTS][ncta][BLK], pushed by the CTAs
    const uint32_t push_bytes = ncta * BLK * (uint32_t)sizeof(float2);  // per slot and block
    const float inv_cols = 1.0f / (float)cols;
    const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(gamma + col));
    const float2 g2[4] = {bf16x2_f2(gv.x), bf16x2_f2(gv.y), bf16x2_f2(gv.z), bf16x2_f2(gv.w)};
    const int64_t goff0 = (int64_t)(RPT * g) * cols + col;  // element offset of the thread's first row, less r0
    auto issue = [&](int64_t j, int buf) {
        if (j < nb) {
            const int64_t r0 = (cid + j * ncl) * BLK;
            const int64_t goff = goff0 + r0 * cols, lim = rows - r0 - RPT * g;  // row i is valid while i < lim
            uint8_t *b = lsm + buf * BUF;
#pragma unroll
            for (int i = 0; i < RPT; i++) {
                const bool valid = i < lim;
                const int64_t off = valid ? goff + i * cols : 0;
                const int soff = ((RPT * g + i) * LC_COLS + 8 * c) * 2;
                cp_async16(smem_u32(b + soff), dy + off, valid);
                cp_async16(smem_u32(b + BLK * LC_COLS * 2 + soff), x + off, valid);
            }
            if (t < 2 * BLK) {
                const int64_t row = r0 + (t % BLK);
                const bool valid = row < rows;
                cp_async4(smem_u32(&mrs[buf][t / BLK][t % BLK]), (t < BLK ? mu : rs) + (valid ? row : 0), valid);
            }
        }
        cp_async_commit();
    };
    auto drow = [&](int buf) { return reinterpret_cast<const uint4 *>(lsm + buf * BUF + RPT * g * LC_COLS * 2) + c; };
    auto xrow = [&](int buf) {
        return reinterpret_cast<const uint4 *>(lsm + buf * BUF + (BLK + RPT * g) * LC_COLS * 2) + c;
    };
    float2 pg[4], pb[4];  // column partials of dgamma, dbeta (columns 2k, 2k+1 in pg[k])
#pragma unroll
    for (int k = 0; k < 4; k++) pg[k] = pb[k] = make_float2(0.0f, 0.0f);
    // Per-warp row partials of the staged block in `buf` into wsum; column partials into pg/pb.
    auto partials = [&](int buf) {
        const uint4 *dr = drow(buf), *xr = xrow(buf);
        float2 s[RPT];
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const float m = mrs[buf][0][RPT * g + i], sg = mrs[buf][1][RPT * g + i];
            const float2 nm = make_float2(-m, -m), sg2 = make_float2(sg, sg);
            const uint4 dq = dr[i * (LC_COLS / 8)], xq = xr[i * (LC_COLS / 8)];
            const uint32_t dv[4] = {dq.x, dq.y, dq.z, dq.w}, xv[4] = {xq.x, xq.y, xq.z, xq.w};
            float2 s1 = make_float2(0.0f, 0.0f), s2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float2 d = bf16x2_f2(dv[q]);
                const float2 h = __fmul2_rn(__fadd2_rn(bf16x2_f2(xv[q]), nm), sg2);  // xhat
                const float2 gg = __fmul2_rn(d, g2[q]);                              // dy * gamma
                s1 = __fadd2_rn(s1, gg);
                s2 = __ffma2_rn(gg, h, s2);
                pg[q] = __ffma2_rn(d, h, pg[q]);
                pb[q] = __fadd2_rn(pb[q], d);
            }
            s[i] = make_float2(s1.x + s1.y, s2.x + s2.y);
        }
        const float2 r = warp_sum_rows<RPT>(s, lane);
        if ((lane & (32 / RPT - 1)) == 0) wsum[w][lane / (32 / RPT)] = r;
    };
    // After a barrier: the CTA's row partials from the two warps of each row group, pushed into
    // slot `slot` of every CTA of the cluster (this CTA's entry), completing on that CTA's barrier.
    auto push = [&](int slot) {
        if (t < BLK) {
            const float2 a = wsum[2 * (t / RPT)][t % RPT], b = wsum[2 * (t / RPT) + 1][t % RPT];
            const float2 v = make_float2(a.x + b.x, a.y + b.y);
            const uint32_t la = smem_u32(&gath[(slot * ncta + rank) * BLK + t]), lb = smem_u32(&xbar[slot]);
            for (uint32_t k = 0; k < ncta; k++) st_async_f2(mapa_shared(la, k), v, mapa_shared(lb, k));
        }
    };
    if (t == 0) {
        for (int k = 0; k < LC_SLOTS; k++) mbar_init(smem_u32(&xbar[k]), 1);
        mbar_fence_init();
    }
    cluster_sync();  // every CTA's barriers are initialised before anything is pushed to them
    if (t == 0)
        for (int k = 0; k < LC_SLOTS && k < nb; k++) mbar_expect_tx(smem_u32(&xbar[k]), push_bytes);
    if (nb > 0) {  // always, as no more clusters than blocks are launched
        issue(0, 0);
        issue(1, 1);
        cp_async_wait<1>();
        __syncthreads();  // mu and rs of block 0 were copied by other threads
        partials(0);
        __syncthreads();
        push(0);
    }
    int buf = 0, slot = 0;
    for (int64_t j = 0; j < nb; j++) {
        const int64_t r0 = (cid + j * ncl) * BLK;
        const int nslot = (slot + 1) & (LC_SLOTS - 1);
        cp_async_wait<0>();  // block j+1 has landed (the only group in flight)
        __syncthreads();     // ... including mu and rs; every thread is past block j-1
        issue(j + 2, next_buf(next_buf(buf)));
        // block j+1's partials are pushed before block j is gathered: with short blocks the
        // pushes of block j then have a whole reduction to arrive in
        if (j + 1 < nb) {
            partials(next_buf(buf));
            __syncthreads();
            push(nslot);
        }
        if (t >= 32 && t < 32 + BLK) {  // warp 1 gathers while warp 0 pushes
            const int r = t - 32;
            // every CTA's partials of block j have arrived (a wait that runs out leaves NaN)
            const bool arrived = mbar_wait_bounded(smem_u32(&xbar[slot]), (uint32_t)((j / LC_SLOTS) & 1));
            const float nan = __int_as_float(0x7fc00000);
            float2 tot = arrived ? make_float2(0.0f, 0.0f) : make_float2(nan, nan);
            for (uint32_t k = 0; k < ncta; k++) {  // rank order
                const float2 p = gath[(slot * ncta + k) * BLK + r];
                tot.x += p.x;
                tot.y += p.y;
            }
            cst[r] = make_float2(tot.x * inv_cols, tot.y * inv_cols);
            // the slot's next block: its barrier counts the pushes of block j + LC_SLOTS
            if (r == 0 && j + LC_SLOTS < nb) mbar_expect_tx(smem_u32(&xbar[slot]), push_bytes);
        }
        __syncthreads();
        if (r0 + RPT * g < rows) {  // rows are a multiple of 16: always
            const uint4 *dr = drow(buf), *xr = xrow(buf);
#pragma unroll
            for (int i = 0; i < RPT; i++) {
                const float2 cc = cst[RPT * g + i];
                const float m = mrs[buf][0][RPT * g + i], sg = mrs[buf][1][RPT * g + i];
                const float2 nm = make_float2(-m, -m), sg2 = make_float2(sg, sg);
                const float k1 = -sg * cc.x, k2 = -(sg * sg) * cc.y;
                const uint4 dq = dr[i * (LC_COLS / 8)], xq = xr[i * (LC_COLS / 8)];
                const uint32_t dv[4] = {dq.x, dq.y, dq.z, dq.w}, xv[4] = {xq.x, xq.y, xq.z, xq.w};
                uint32_t ow[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    // dx = (x - mu) * k2 + (rs * (dy * gamma) + k1), two at a time
                    const float2 u = __ffma2_rn(__fmul2_rn(bf16x2_f2(dv[q]), g2[q]), sg2, f2(k1));
                    ow[q] = f2_bf16x2(__ffma2_rn(__fadd2_rn(bf16x2_f2(xv[q]), nm), f2(k2), u));
                }
                *reinterpret_cast<uint4 *>(dx + goff0 + (r0 + i) * cols) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
        }
        buf = next_buf(buf);
        slot = nslot;
    }
    cp_async_wait<0>();
    __syncthreads();  // every thread is done with the staged blocks: reuse them for the column partials
    float *red = reinterpret_cast<float *>(lsm);  // [dgamma, dbeta][row group][LC_COLS]
    {
        float4 *dg4 = reinterpret_cast<float4 *>(red + (0 * 4 + g) * LC_COLS + 8 * c);
        float4 *db4 = reinterpret_cast<float4 *>(red + (1 * 4 + g) * LC_COLS + 8 * c);
        dg4[0] = make_float4(pg[0].x, pg[0].y, pg[1].x, pg[1].y);
        dg4[1] = make_float4(pg[2].x, pg[2].y, pg[3].x, pg[3].y);
        db4[0] = make_float4(pb[0].x, pb[0].y, pb[1].x, pb[1].y);
        db4[1] = make_float4(pb[2].x, pb[2].y, pb[3].x, pb[3].y);
    }
    __syncthreads();
    for (int k = t; k < LC_COLS; k += LC_THREADS) {
        float a = red[k], b = red[4 * LC_COLS + k];
#pragma unroll
        for (int q = 1; q < 4; q++) {
            a += red[q * LC_COLS + k];
            b += red[(4 + q) * LC_COLS + k];
        }
        part[cid * cols + col0 + k] = a;
        part[(ncl + cid) * cols + col0 + k] = b;
    }
    cluster_sync();  // every push to this CTA has arrived (it waited for them); none leaves before the rest
}

// ---------------------------------------------------------------------------
// Host side of the cluster path.
// ---------------------------------------------------------------------------
// Cluster size for `cols`, or 0 when the cluster path does not apply.
static int ln_cluster_size(int64_t cols) {
    return (cols % LC_COLS == 0 && cols / LC_COLS <= LC_MAX_CLUSTER) ? (int)(cols / LC_COLS) : 0;
}

static void cluster_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *at, int64_t clusters, int cl, int smem,
                           cudaStream_t st) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3((unsigned)(clusters * cl), 1, 1);
    cfg.blockDim = dim3(LC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cl;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
}

// How many clusters of `cl` CTAs of `kernel` can be resident at once (0: none).
static int ln_max_clusters(const void *kernel, int smem, int smem_max, int cl) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e == cudaSuccess && cl > 8) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute at[1];
    cluster_config(cfg, at, 1, cl, smem, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    return n;
}

// Resident-cluster counts + 1 per device, kernel (0 fwd E4M3, 1 fwd E5M2, 2 bwd) and cluster
// size; 0 = not queried yet.
static std::atomic<int> g_ln_clusters[64][3][LC_MAX_CLUSTER + 1];

// Number of clusters to launch over `nblk` row blocks, or 0 to take the tile path.
// FP8DL_LN_VARIANT=tiles forces the tile path and FP8DL_LN_CLUSTERS=n caps the
// cluster count (both for testing).
static int64_t ln_cluster_count(int dev, int which, const void *kernel, int smem_base, int slot_rows, int64_t nblk,
                                int64_t cols, int64_t cap) {
    const char *v = getenv("FP8DL_LN_VARIANT");
    if (v && v[0] == 't') return 0;
    const int cl = ln_cluster_size(cols);
    if (cl == 0) return 0;
    std::atomic<int> &slot = g_ln_clusters[dev][which][cl];
    int known = slot.load(std::memory_order_acquire);
    if (known == 0) {
        std::lock_guard<std::mutex> lock(init_mutex());
        known = slot.load(std::memory_order_relaxed);
        if (known == 0) {
            // sets the kernel's attributes first (shared memory for the largest cluster)
            known = ln_max_clusters(kernel, ln_smem(smem_base, slot_rows, cl),
                                    ln_smem(smem_base, slot_rows, LC_MAX_CLUSTER), cl) + 1;
            slot.store(known, std::memory_order_release);
        }
    }
    const int64_t resident = known - 1;
    if (resident <= 0) return 0;
    int64_t n = nblk < resident ? nblk : resident;
    if (n > cap) n = cap;
    const char *lim = getenv("FP8DL_LN_CLUSTERS");
    if (lim && atoll(lim) > 0 && n > atoll(lim)) n = atoll(lim);
    return n;
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_clustered(void (*kernel)(KArgs...), int64_t clusters, int cl, int smem, cudaStream_t st, bool pdl,
                                    Args... args) {
    const cudaError_t e = launch_kernel(kernel, dim3((unsigned)(clusters * cl)), dim3(LC_THREADS), (size_t)smem, st,
                                        cl, pdl, args...);
    if (e == cudaSuccess) note_launch();
    return e;
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
    const bool pdl = short_call_bytes((double)rows * cols * 4);
    auto X = static_cast<const uint16_t *>(x);
    {
        const bool e4 = out_dtype == FP8DL_E4M3;
        auto kern = e4 ? ln_fwd_cluster_kernel<FP8DL_E4M3> : ln_fwd_cluster_kernel<FP8DL_E5M2>;
        const int64_t ncl = ln_cluster_count(dev, e4 ? 0 : 1, (const void *)kern, LF_SMEM, LF_ROWS,
                                              (rows + LF_ROWS - 1) / LF_ROWS, cols, INT64_MAX);
        if (ncl > 0) {
            const int cl = ln_cluster_size(cols);
            const cudaError_t e = launch_clustered(kern, ncl, cl, ln_smem(LF_SMEM, LF_ROWS, cl), st, pdl, X,
                                                   static_cast<const uint16_t *>(gamma),
                                                   static_cast<const uint16_t *>(beta), rows, cols, eps, scale, out,
                                                   out_t, amax, mu, rsigma, static_cast<uint16_t *>(y));
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(FP8DL_ERR_CUDA, "fp8_layernorm_cast(cluster): %s", cudaGetErrorString(e));
            }
            return check_launch("fp8_layernorm_cast(cluster)");
        }
    }
    // tile path. pass 1: per-row statistics (one read of x); pass 2: normalise + cast in 128x128 tiles
    const int64_t chunks_per_lane = (cols / 8 + 31) / 32;
    const int64_t row_ctas = (rows + 7) / 8;
    const unsigned g1 = (unsigned)(row_ctas < (int64_t)sms * 8 ? row_ctas : (int64_t)sms * 8);
    if (chunks_per_lane <= 4)
        (void)launch_kernel(ln_stats_kernel<4>, g1, 256, 0, st, 0, pdl, X, rows, cols, eps, mu, rsigma);
    else if (chunks_per_lane <= 8)
        (void)launch_kernel(ln_stats_kernel<8>, g1, 256, 0, st, 0, pdl, X, rows, cols, eps, mu, rsigma);
    else if (chunks_per_lane <= 16)
        (void)launch_kernel(ln_stats_kernel<16>, g1, 256, 0, st, 0, pdl, X, rows, cols, eps, mu, rsigma);
    else
        (void)launch_kernel(ln_stats_kernel<32>, g1, 256, 0, st, 0, pdl, X, rows, cols, eps, mu, rsigma);
    note_launch();
    FP8DL_TRY(check_launch("fp8_layernorm_cast(statistics)"));
    if (!(out || out_t || amax || y)) return FP8DL_OK;
    return launch_layernorm_tile_cast(x, mu, rsigma, gamma, beta, rows, cols, out_dtype, scale, out, out_t, amax, y,
                                      sms, st, pdl);
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
    int dev = 0, sms = 0;
    FP8DL_TRY(current_device(&dev, &sms));
    cudaStream_t st = (cudaStream_t)stream;
    const bool pdl = short_call_bytes((double)rows * cols * 6);
    float *c12 = static_cast<float *>(workspace);
    float *part = c12 + 2 * rows;
    auto DY = static_cast<const uint16_t *>(dy);
    auto X = static_cast<const uint16_t *>(x);
    auto G = static_cast<const uint16_t *>(gamma);
    const int64_t n_rt = (rows + LB_ROWS - 1) / LB_ROWS;
    {
        // the workspace holds n_rt partial rows per output: at most n_rt clusters
        const int64_t ncl = ln_cluster_count(dev, 2, (const void *)ln_bwd_cluster_kernel<LB_BLK>, LB_SMEM, LB_BLK,
                                              (rows + LB_BLK - 1) / LB_BLK, cols, n_rt);
        if (ncl > 0) {
            const int cl = ln_cluster_size(cols);
            const cudaError_t e = launch_clustered(ln_bwd_cluster_kernel<LB_BLK>, ncl, cl, ln_smem(LB_SMEM, LB_BLK, cl), st, pdl,
                                                   DY, X, G, mu, rsigma, rows, cols, static_cast<uint16_t *>(dx), part);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(FP8DL_ERR_CUDA, "fp8_layernorm_bwd(cluster): %s", cudaGetErrorString(e));
            }
            FP8DL_TRY(check_launch("fp8_layernorm_bwd(cluster)"));
            (void)launch_kernel(ln_bwd_reduce_kernel, (unsigned)((cols + 31) / 32), 256, 0, st, 0, pdl, part, ncl, cols, dgamma, dbeta);
            note_launch();
            return check_launch("fp8_layernorm_bwd(reduce)");
        }
    }
    const int64_t row_ctas = (rows + 7) / 8;
    (void)launch_kernel(ln_bwd_rowsum_kernel, (unsigned)(row_ctas < (int64_t)sms * 8 ? row_ctas : (int64_t)sms * 8), 256, 0, st, 0, pdl, 
        DY, X, G, mu, rsigma, rows, cols, c12);
    note_launch();
    FP8DL_TRY(check_launch("fp8_layernorm_bwd(row sums)"));
    const int64_t tiles = n_rt * ((cols + LB_COLS - 1) / LB_COLS);
    (void)launch_kernel(ln_bwd_tile_kernel, (unsigned)(tiles < (int64_t)sms * 4 ? tiles : (int64_t)sms * 4), 256, 0, st, 0, pdl, 
        DY, X, G, mu, rsigma, c12, rows, cols, static_cast<uint16_t *>(dx), part);
    note_launch();
    FP8DL_TRY(check_launch("fp8_layernorm_bwd(dx)"));
    (void)launch_kernel(ln_bwd_reduce_kernel, (unsigned)((cols + 31) / 32), 256, 0, st, 0, pdl, part, n_rt, cols, dgamma, dbeta);
    note_launch();
    return check_launch("fp8_layernorm_bwd(reduce)");
}

}  // extern "C"
