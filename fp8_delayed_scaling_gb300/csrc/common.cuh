// common.cuh — shared host/device helpers of the fp8dl library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "fp8dl.h"
#include <nvtx3/nvToolsExt.h>

namespace fp8dl {

// ---------------------------------------------------------------------------
// Host-side error reporting: a thread-local message and a status code.
// ---------------------------------------------------------------------------
void set_error(const char *fmt, ...);
fp8dl_status fail(fp8dl_status st, const char *fmt, ...);
fp8dl_status check_launch(const char *what);

// Counts one kernel launch of this library (read through fp8dl_kernel_launches).
void note_launch();

// Serialises the library's one-time, per-device set-up (function attributes, occupancy
// queries, symbol addresses) across host threads.  The caches it fills are atomics read
// with acquire ordering, so a thread that sees a cache entry also sees what it stands for.
std::mutex &init_mutex();

// Validates the current device (sm_103) once per device and caches the SM count.
fp8dl_status current_device(int *dev, int *num_sms);

// dbias[c] = sum over r of ws[r * cols + c] (fp32, a fixed order), one launch on st
// (programmatic when `pdl`: the calling ABI call is a short one).
void colsum_reduce(const float *ws, int64_t n_rows, int64_t cols, float *dbias, cudaStream_t st, bool pdl);

// An NVTX range over one ABI call (visible to nsys/ncu; nearly free without a tool).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};
#define FP8DL_NVTX(name) ::fp8dl::NvtxRange fp8dl_nvtx_range_(name)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool dim_ok(int64_t d, int64_t mult) { return d > 0 && d % mult == 0 && d <= (int64_t(1) << 31); }

#define FP8DL_CHECK_ARG(cond, ...)                                                                \
    do {                                                                                          \
        if (!(cond)) return ::fp8dl::fail(FP8DL_ERR_INVALID_ARG, __VA_ARGS__);                    \
    } while (0)

#define FP8DL_TRY(expr)                                                                           \
    do {                                                                                          \
        fp8dl_status _s = (expr);                                                                 \
        if (_s != FP8DL_OK) return _s;                                                            \
    } while (0)

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The library launches the kernels of short
// calls (short_call_bytes / short_call_flops below) with the programmatic
// stream serialization attribute (unless FP8DL_PDL=0), so such a kernel may
// start while the previous kernel of its stream is still running: its
// launch and set-up (barrier initialisation, tensor-memory allocation,
// descriptor prefetch) overlap that kernel's tail.  pdl_wait() blocks until the
// previous kernel has completed and its memory operations are visible; every
// kernel calls it before its first access to global memory.  pdl_trigger()
// lets the next kernel begin launching once every CTA of this one has called it
// or exited (it then waits in its own pdl_wait()).  Both are no-ops in a kernel
// launched without the attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// FP8DL_PDL unset or not "0" (read once per process).
bool pdl_enabled();

// Which launches take the attribute: short ones, whose launch latency and set-up
// are a visible part of their time (an ABI call moving under 64 MB or doing
// under 64 GFLOP, tens of microseconds).  Measured on the step workloads: the
// te.Linear layer (2048 x 768 -> 3072) ran 7 % faster with every launch
// programmatic, while the LayerNormMLP and Llama blocks, whose kernels run
// hundreds of microseconds, ran about 2 % slower.
inline bool short_call_bytes(double bytes) { return bytes < 64.0 * 1024 * 1024; }
inline bool short_call_flops(double flops) { return flops < 64e9; }

// kernel<<<grid, block, smem, st>>>(args...) through cudaLaunchKernelEx, with the
// programmatic serialization attribute when `pdl` and enabled.  cluster = 0: no cluster
// attribute (a kernel with __cluster_dims__ keeps its own); cluster >= 1: a
// cluster of that many CTAs along x, also for 1 (a kernel that uses cluster
// shared memory or cluster barriers must be launched as a cluster, even of one
// CTA).  A launch error is also left for cudaGetLastError (check_launch).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          int cluster, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    unsigned n = 0;
    if (pdl && pdl_enabled()) {
        at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[n].val.programmaticStreamSerializationAllowed = 1;
        n++;
    }
    if (cluster >= 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = (unsigned)cluster;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        n++;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Device-side FP8 conversion through the hardware cvt (round to nearest even,
// saturating to the largest finite value; NaN stays NaN).
// cvt.rn.satfinite.{e4m3x2,e5m2x2}.f32 d, a, b packs a into the high byte.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t cvt_e5m2x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 values -> four codes packed little-endian (v0 in byte 0).
template <int FMT>
__device__ __forceinline__ uint32_t pack4(float v0, float v1, float v2, float v3) {
    uint32_t lo, hi;
    if (FMT == FP8DL_E4M3) {
        lo = cvt_e4m3x2(v1, v0);
        hi = cvt_e4m3x2(v3, v2);
    } else {
        lo = cvt_e5m2x2(v1, v0);
        hi = cvt_e5m2x2(v3, v2);
    }
    return lo | (hi << 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// |a| and |b| maxima of two bf16x2 words, lane by lane (the sign bits of the
// result are the XOR of the inputs' and carry no meaning; a NaN input is
// ignored, as fmaxf ignores it).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Non-negative floats order like their bit patterns: atomicMax on the bits.
__device__ __forceinline__ void atomic_max_nonneg(float *addr, float v) {
    atomicMax(reinterpret_cast<unsigned int *>(addr), __float_as_uint(v));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Streaming 16-byte global load that bypasses L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// Activation math shared by the cast kernels and the GEMM epilogue.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ float ex2_approx_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The erf GELU, GELU(h) = h * Phi(h) with Phi the standard normal CDF, and its
// derivative GELU'(h) = Phi(h) + h * phi(h), phi the density.  Both take the
// lower tail T(h) = Phi(-|h|) from Abramowitz & Stegun, Handbook of
// Mathematical Functions, formula 26.2.17: for x >= 0
//   Phi(-x) = phi(x) * (b1 t + b2 t^2 + b3 t^3 + b4 t^4 + b5 t^5) + eps,
//   t = 1 / (1 + p x),  |eps| < 7.5e-8,
// with the density's factor 1/sqrt(2 pi) folded into the b's and
// exp(-h^2/2) = 2^(-h^2 log2(e) / 2) from the hardware approximations (total
// |dPhi| < 3e-7).  Flushing a subnormal exponential to zero (|h| > 13) changes
// a result by less than |h| * 2^-126.
struct NormalTail {
    float e;     // exp(-h^2 / 2)
    float tail;  // Phi(-|h|)
};
__device__ __forceinline__ NormalTail normal_tail(float h) {
    constexpr float K = 0.3989422804f;  // 1 / sqrt(2 pi)
    const float e = ex2_approx_ftz(h * h * -0.7213475204f);
    const float t = rcp_approx_ftz(fmaf(0.2316419f, fabsf(h), 1.0f));
    float poly = fmaf(t, 1.330274429f * K, -1.821255978f * K);
    poly = fmaf(t, poly, 1.781477937f * K);
    poly = fmaf(t, poly, -0.356563782f * K);
    poly = fmaf(t, poly, 0.319381530f * K);
    return {e, e * poly * t};
}

// GELU(h) in fp32 (before the bf16 rounding), written as
//   GELU(h) = max(h, 0) - |h| * Phi(-|h|),
// which is h * (1 - Phi(-h)) for h >= 0 and h * Phi(h) for h < 0: one fused
// multiply-add instead of a select.
__device__ __forceinline__ float gelu_f32(float h) {
    return fmaf(-fabsf(h), normal_tail(h).tail, fmaxf(h, 0.0f));
}

// GELU(h) rounded to bf16 like the tensor it stands for.
__device__ __forceinline__ float gelu_bf16(float h) { return bf16_round(gelu_f32(h)); }

// dh = dg * GELU'(h) = dg * (Phi(h) + h * phi(h)) in fp32, and rounded to bf16.
__device__ __forceinline__ float dgelu_f32(float dg, float h) {
    const NormalTail n = normal_tail(h);
    const float cdf = h >= 0.0f ? 1.0f - n.tail : n.tail;
    return dg * fmaf(h * 0.3989422804f, n.e, cdf);
}
__device__ __forceinline__ float dgelu_bf16(float dg, float h) { return bf16_round(dgelu_f32(dg, h)); }

// The same three functions on two values at once with fp32x2 instructions (half the
// issue slots).  Each lane runs the scalar form's operations in the same order with the
// same rounding, so the results are bit-identical to gelu_f32 / dgelu_f32.  The tail
// comes out negated: every coefficient of the polynomial is negated, which is exact
// because round-to-nearest is symmetric, and -|h| * T becomes |h| * (-T).
struct NormalTail2 {
    float2 e;      // exp(-h^2 / 2)
    float2 ntail;  // -Phi(-|h|)
};
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }
__device__ __forceinline__ NormalTail2 normal_tail2(float2 h, float2 ah) {
    constexpr float K = 0.3989422804f;
    const float2 a = __fmul2_rn(__fmul2_rn(h, h), f2(-0.7213475204f));
    const float2 e = make_float2(ex2_approx_ftz(a.x), ex2_approx_ftz(a.y));
    const float2 d = __ffma2_rn(f2(0.2316419f), ah, f2(1.0f));
    const float2 t = make_float2(rcp_approx_ftz(d.x), rcp_approx_ftz(d.y));
    float2 poly = __ffma2_rn(t, f2(-1.330274429f * K), f2(1.821255978f * K));
    poly = __ffma2_rn(t, poly, f2(-1.781477937f * K));
    poly = __ffma2_rn(t, poly, f2(0.356563782f * K));
    poly = __ffma2_rn(t, poly, f2(-0.319381530f * K));
    return {e, __fmul2_rn(__fmul2_rn(e, poly), t)};
}
__device__ __forceinline__ float2 gelu2_f32(float2 h) {
    const float2 ah = make_float2(fabsf(h.x), fabsf(h.y));
    return __ffma2_rn(ah, normal_tail2(h, ah).ntail, make_float2(fmaxf(h.x, 0.0f), fmaxf(h.y, 0.0f)));
}
__device__ __forceinline__ float2 dgelu2_f32(float2 dg, float2 h) {
    const NormalTail2 n = normal_tail2(h, make_float2(fabsf(h.x), fabsf(h.y)));
    const float2 omt = __fadd2_rn(f2(1.0f), n.ntail);  // 1 - Phi(-|h|)
    const float2 cdf = make_float2(h.x >= 0.0f ? omt.x : -n.ntail.x, h.y >= 0.0f ? omt.y : -n.ntail.y);
    return __fmul2_rn(dg, __ffma2_rn(__fmul2_rn(h, f2(0.3989422804f)), n.e, cdf));
}


}  // namespace fp8dl
