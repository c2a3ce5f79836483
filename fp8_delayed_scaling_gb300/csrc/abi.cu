// abi.cu — library state of the C ABI: error messages, device checks, version.
#include <stdarg.h>
#include <atomic>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"

namespace fp8dl {

static thread_local char g_last_error[512] = "";

static bool debug_enabled() {
    static int flag = -1;
    if (flag < 0) {
        const char *e = getenv("FP8DL_DEBUG");
        flag = (e && e[0] && e[0] != '0') ? 1 : 0;
    }
    return flag == 1;
}

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    if (debug_enabled()) fprintf(stderr, "[fp8dl] %s\n", g_last_error);
}

fp8dl_status fail(fp8dl_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    if (debug_enabled()) fprintf(stderr, "[fp8dl] error %d: %s\n", (int)st, g_last_error);
    return st;
}

std::atomic<uint64_t> g_launches{0};

bool pdl_enabled() {
    static const bool on = [] {
        const char *e = getenv("FP8DL_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

// One record per CTA: the SM it ran on, that SM's cycle counter and the global
// nanosecond timer, read together by lane 0.
__global__ void clock_probe_kernel(uint64_t *__restrict__ out) {
    if (threadIdx.x != 0) return;
    uint32_t smid;
    uint64_t ns;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const long long c = clock64();
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
    out[3 * blockIdx.x] = smid;
    out[3 * blockIdx.x + 1] = (uint64_t)c;
    out[3 * blockIdx.x + 2] = ns;
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

fp8dl_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP8DL_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    if (debug_enabled()) fprintf(stderr, "[fp8dl] launched %s\n", what);
    return FP8DL_OK;
}

std::mutex &init_mutex() {
    static std::mutex m;
    return m;
}

// Per-device cache: 0 = unknown, 1 = supported, -1 = unsupported (g_dev_sms is written first).
static std::atomic<int> g_dev_state[64];
static int g_dev_sms[64];

static int probe_device(int dev) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (dev >= 0 && dev < 64) g_dev_sms[dev] = sms;
    return (major == 10 && minor == 3) ? 1 : -1;
}

fp8dl_status current_device(int *dev, int *num_sms) {
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return fail(FP8DL_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (d < 0 || d >= 64) return fail(FP8DL_ERR_UNSUPPORTED_DEVICE, "device index %d out of range", d);
    int st = g_dev_state[d].load(std::memory_order_acquire);
    if (st == 0) {
        std::lock_guard<std::mutex> lock(init_mutex());
        st = g_dev_state[d].load(std::memory_order_relaxed);
        if (st == 0) {
            st = probe_device(d);
            g_dev_state[d].store(st, std::memory_order_release);
        }
    }
    if (st != 1) return fail(FP8DL_ERR_UNSUPPORTED_DEVICE, "device %d is not an sm_103 (GB300) GPU", d);
    if (dev) *dev = d;
    if (num_sms) *num_sms = g_dev_sms[d];
    return FP8DL_OK;
}

}  // namespace fp8dl

extern "C" {

const char *fp8dl_last_error(void) { return fp8dl::g_last_error; }

int32_t fp8dl_version(void) { return 100; }

uint64_t fp8dl_kernel_launches(void) { return fp8dl::g_launches.load(std::memory_order_relaxed); }

fp8dl_status fp8dl_clock_probe(uint64_t *out, int32_t n_ctas, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8dl_clock_probe");
    FP8DL_CHECK_ARG(out != nullptr, "out is NULL");
    FP8DL_CHECK_ARG(n_ctas >= 1 && n_ctas <= 65536, "n_ctas must be in [1, 65536]");
    if (!fp8dl::aligned16(out)) return fp8dl::fail(FP8DL_ERR_ALIGN, "out must be 16-byte aligned");
    FP8DL_TRY(fp8dl::current_device(nullptr, nullptr));
    fp8dl::clock_probe_kernel<<<(unsigned)n_ctas, 32, 0, (cudaStream_t)stream>>>(out);
    fp8dl::note_launch();
    return fp8dl::check_launch("fp8dl_clock_probe");
}

int32_t fp8dl_device_supported(int32_t device) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (device < 0 || device >= n || device >= 64) return 0;
    return fp8dl::probe_device(device) == 1 ? 1 : 0;
}

}  // extern "C"
