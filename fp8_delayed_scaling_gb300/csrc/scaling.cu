// scaling.cu — delayed-scaling state: init, amax-history update, first-step seeding.
//
// "FP8 低精度训练：Transformer Engine 简析", §三.1 "宏观实现框架": each scaled
// tensor keeps an amax history; the maximum over the window stands in for the
// tensor's amax and the scale is (FP8_MAX / amax) / 2^margin; `interval` sets
// how often the scale is recomputed.  §三.3: the update runs when the step's
// casts have recorded their amaxes (autocast exit), so the new scale is used by
// the next step's casts — the delay that gives the method its name.
#include "common.cuh"

namespace fp8dl {

struct SlotHeader {
    float scale;
    float scale_inv;
    float amax;
    int32_t hist_pos;
    int32_t fp8_dtype;
    int32_t reserved[3];
};
static_assert(sizeof(SlotHeader) == 32, "slot header is 32 bytes");

static inline int64_t hist_padded(int32_t L) { return (int64_t(L) + 3) / 4 * 4; }

__device__ __forceinline__ SlotHeader *slot_at(void *state, int64_t stride, int i) {
    return reinterpret_cast<SlotHeader *>(static_cast<char *>(state) + stride * i);
}

__device__ __forceinline__ float fp8_max_of(int dtype) { return dtype == FP8DL_E5M2 ? 57344.0f : 448.0f; }

// scale = fl32(FP8_MAX / a) / 2^margin; kept unless a and the result are finite and positive.
__device__ __forceinline__ void recompute(SlotHeader *h, float a, int margin) {
    if (!(a > 0.0f) || isinf(a)) return;
    float s = __fdiv_rn(fp8_max_of(h->fp8_dtype), a);
    const float p = __int_as_float((margin + 127) << 23);  // 2^margin, exact for 0..126
    s = __fdiv_rn(s, p);
    if (!(s > 0.0f) || isinf(s)) return;
    h->scale = s;
    h->scale_inv = __frcp_rn(s);
}

// One warp per slot.
__global__ void update_scale_kernel(void *state, int64_t stride, int n_slots, int L, int margin,
                                    int do_recompute, int seed) {
    pdl_wait();  // the previous kernel of the stream has completed
    pdl_trigger();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= n_slots) return;
    SlotHeader *h = slot_at(state, stride, warp);
    float *hist = reinterpret_cast<float *>(h + 1);
    const float cur = h->amax;
    if (seed) {
        for (int i = lane; i < L; i += 32) hist[i] = cur;
    } else if (lane == 0) {
        int pos = h->hist_pos;
        hist[pos] = cur;
    }
    __syncwarp();
    float m = 0.0f;
    for (int i = lane; i < L; i += 32) m = fmaxf(m, hist[i]);
    m = warp_max(m);
    if (lane == 0) {
        h->hist_pos = seed ? 0 : (h->hist_pos + 1) % L;
        h->amax = 0.0f;
        if (do_recompute) recompute(h, m, margin);
    }
}

struct InitMask {
    uint32_t e5m2[32];  // bit i of word w: slot (32*w + i) of this launch is E5M2
};

__global__ void init_state_kernel(void *state, int64_t stride, int first, int count, int Lp, InitMask mask) {
    const int s = blockIdx.x;
    if (s >= count) return;
    SlotHeader *h = slot_at(state, stride, first + s);
    float *hist = reinterpret_cast<float *>(h + 1);
    for (int i = threadIdx.x; i < Lp; i += blockDim.x) hist[i] = 0.0f;
    if (threadIdx.x == 0) {
        h->scale = 1.0f;
        h->scale_inv = 1.0f;
        h->amax = 0.0f;
        h->hist_pos = 0;
        h->fp8_dtype = ((mask.e5m2[s >> 5] >> (s & 31)) & 1u) ? FP8DL_E5M2 : FP8DL_E4M3;
        h->reserved[0] = h->reserved[1] = h->reserved[2] = 0;
    }
}

static fp8dl_status check_recipe(const fp8dl_recipe *r, int32_t n_slots, const void *state) {
    FP8DL_CHECK_ARG(r != nullptr, "recipe is NULL");
    FP8DL_CHECK_ARG(state != nullptr, "state is NULL");
    FP8DL_CHECK_ARG(n_slots >= 1, "n_slots must be >= 1 (got %d)", n_slots);
    FP8DL_CHECK_ARG(r->margin >= 0 && r->margin <= 126, "margin must be in [0, 126] (got %d)", r->margin);
    FP8DL_CHECK_ARG(r->interval >= 1, "interval must be >= 1 (got %d)", r->interval);
    FP8DL_CHECK_ARG(r->amax_history_len >= 1 && r->amax_history_len <= (1 << 20),
                    "amax_history_len must be in [1, 2^20] (got %d)", r->amax_history_len);
    FP8DL_CHECK_ARG(r->amax_compute_algo == 0, "amax_compute_algo: only 0 (max) is defined");
    FP8DL_CHECK_ARG(r->fp8_format == FP8DL_FORMAT_E4M3 || r->fp8_format == FP8DL_FORMAT_HYBRID,
                    "unknown fp8_format %d", r->fp8_format);
    if (!aligned16(state)) return fail(FP8DL_ERR_ALIGN, "state must be 16-byte aligned");
    return FP8DL_OK;
}

static fp8dl_status launch_update(const fp8dl_recipe *recipe, int32_t n_slots, void *state, int64_t step,
                                  int seed, cudaStream_t stream) {
    FP8DL_TRY(check_recipe(recipe, n_slots, state));
    FP8DL_TRY(current_device(nullptr, nullptr));
    FP8DL_CHECK_ARG(step >= 0, "step must be >= 0");
    const int64_t stride = (int64_t)fp8dl_slot_stride(recipe->amax_history_len);
    const int do_recompute = seed ? 1 : (step % recipe->interval == 0);
    const int threads = 256, slots_per_block = threads / 32;
    const int blocks = (n_slots + slots_per_block - 1) / slots_per_block;
    (void)launch_kernel(update_scale_kernel, blocks, threads, 0, stream, 0, true, state, stride, n_slots, recipe->amax_history_len,
                                                        recipe->margin, do_recompute, seed);
    note_launch();
    return check_launch(seed ? "fp8_seed_amax_history" : "fp8_update_scale");
}

}  // namespace fp8dl

using namespace fp8dl;

extern "C" {

size_t fp8dl_slot_stride(int32_t amax_history_len) {
    if (amax_history_len < 1) return 0;
    return sizeof(SlotHeader) + 4 * (size_t)hist_padded(amax_history_len);
}

size_t fp8dl_scaling_state_bytes(int32_t amax_history_len, int32_t n_slots) {
    if (n_slots < 1) return 0;
    return fp8dl_slot_stride(amax_history_len) * (size_t)n_slots;
}

fp8dl_status fp8_scaling_state_init(const fp8dl_recipe *recipe, int32_t n_slots, const int32_t *slot_fp8_dtype,
                                    void *state, fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_scaling_state_init");
    FP8DL_TRY(check_recipe(recipe, n_slots, state));
    FP8DL_CHECK_ARG(slot_fp8_dtype != nullptr, "slot_fp8_dtype is NULL");
    for (int i = 0; i < n_slots; i++)
        FP8DL_CHECK_ARG(slot_fp8_dtype[i] == FP8DL_E4M3 || slot_fp8_dtype[i] == FP8DL_E5M2,
                        "slot %d: unknown fp8 dtype %d", i, slot_fp8_dtype[i]);
    FP8DL_TRY(current_device(nullptr, nullptr));
    const int64_t stride = (int64_t)fp8dl_slot_stride(recipe->amax_history_len);
    const int Lp = (int)hist_padded(recipe->amax_history_len);
    for (int first = 0; first < n_slots; first += 1024) {
        const int count = n_slots - first < 1024 ? n_slots - first : 1024;
        InitMask m = {};
        for (int s = 0; s < count; s++)
            if (slot_fp8_dtype[first + s] == FP8DL_E5M2) m.e5m2[s >> 5] |= 1u << (s & 31);
        init_state_kernel<<<count, 256, 0, (cudaStream_t)stream>>>(state, stride, first, count, Lp, m);
        note_launch();
        FP8DL_TRY(check_launch("fp8_scaling_state_init"));
    }
    return FP8DL_OK;
}

fp8dl_status fp8_update_scale(const fp8dl_recipe *recipe, int32_t n_slots, void *state, int64_t step,
                              fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_update_scale");
    return launch_update(recipe, n_slots, state, step, 0, (cudaStream_t)stream);
}

fp8dl_status fp8_seed_amax_history(const fp8dl_recipe *recipe, int32_t n_slots, void *state,
                                   fp8dl_stream_t stream) {
    FP8DL_NVTX("fp8_seed_amax_history");
    return launch_update(recipe, n_slots, state, 0, 1, (cudaStream_t)stream);
}

}  // extern "C"
