// Host side of the C ABI: split planner, workspace sizing, argument checks,
// device check and the error-word readback.  No device memory is allocated.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "smla.h"
#include "smla_internal.h"

namespace {

// Cost-model coefficients for GB300 (152 SMs: 76 CTA pairs run at once).
// Units are microseconds; see smla_plan_coeffs in smla.h.
constexpr smla_plan_coeffs kGB300Coeffs = {
    /*slots   */ 76.0,
    /*t0      */ 3.0,
    /*c_entry */ 0.02,
    /*c_byte  */ 3.0e-7,
    /*c_merge */ 3.0,
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// Device check, cached per device (thread-safe).
std::atomic<int> g_dev_ok[64];  // 0 unknown, 1 sm_103, 2 other

smla_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return SMLA_ERR_UNSUPPORTED_DEVICE;
    int state = g_dev_ok[dev].load(std::memory_order_acquire);
    if (state == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SMLA_ERR_CUDA;
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_ok[dev].store(state, std::memory_order_release);
    }
    return state == 1 ? SMLA_OK : SMLA_ERR_UNSUPPORTED_DEVICE;
}

}  // namespace

namespace smla {

smla_status check_decode_args(const smla_decode_args* a) {
    if (a == nullptr) return SMLA_ERR_NULL_POINTER;
    if (a->num_rows < 1 || a->num_rows > SMLA_MAX_ROWS || a->num_heads < 1 || a->num_heads > SMLA_MAX_HEADS ||
        a->num_splits < 1 || a->num_splits > SMLA_MAX_SPLITS || a->topk < 0 || a->n_main < 0 || a->n_cmp < 0 ||
        !std::isfinite(a->sm_scale))
        return SMLA_ERR_BAD_SHAPE;
    if (a->q_nope == nullptr || a->q_rope == nullptr || a->out == nullptr) return SMLA_ERR_NULL_POINTER;
    const bool uses_main = a->topk > 0 || a->swa_len != nullptr;
    if (a->topk > 0 && a->main_idx == nullptr) return SMLA_ERR_NULL_POINTER;
    if (a->swa_len != nullptr && a->swa_start == nullptr) return SMLA_ERR_NULL_POINTER;
    if (uses_main && (a->kv_pool == nullptr || a->kv_scales == nullptr)) return SMLA_ERR_NULL_POINTER;
    if (a->block_table != nullptr && a->pages_per_seq < 1) return SMLA_ERR_BAD_SHAPE;
    if (a->cmp_len != nullptr && (a->cmp_start == nullptr || a->cmp_pool == nullptr || a->cmp_scales == nullptr))
        return SMLA_ERR_NULL_POINTER;
    if (!aligned(a->q_nope, 16) || !aligned(a->q_rope, 16) || !aligned(a->out, 16) ||
        !aligned(a->kv_pool, 16) || !aligned(a->cmp_pool, 16) || !aligned(a->kv_scales, 8) ||
        !aligned(a->cmp_scales, 8) || !aligned(a->block_table, 4) || !aligned(a->row_seq, 4) ||
        !aligned(a->main_idx, 4) || !aligned(a->swa_start, 4) || !aligned(a->swa_len, 4) ||
        !aligned(a->cmp_start, 4) || !aligned(a->cmp_len, 4) || !aligned(a->sink, 4) ||
        !aligned(a->lse, 4))
        return SMLA_ERR_MISALIGNED;
    return SMLA_OK;
}

smla_status check_device_only() { return check_device(); }

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

smla_status check_decode_call(const smla_decode_args* a, const void* workspace, size_t ws_bytes) {
    if (a == nullptr || workspace == nullptr) return SMLA_ERR_NULL_POINTER;
    const smla_status st = check_decode_args(a);
    if (st != SMLA_OK) return st;
    if (!aligned(workspace, 256)) return SMLA_ERR_MISALIGNED;
    if (ws_bytes < smla_workspace_bytes(a->num_rows, a->num_heads, a->num_splits))
        return SMLA_ERR_WORKSPACE_TOO_SMALL;
    return check_device();
}

}  // namespace smla

extern "C" {

smla_status smla_plan_default_coeffs(smla_plan_coeffs* out) {
    if (out == nullptr) return SMLA_ERR_NULL_POINTER;
    *out = kGB300Coeffs;
    return SMLA_OK;
}

int smla_plan_num_splits_ex(int num_rows, int num_heads, int64_t kv_len,
                            const smla_plan_coeffs* coeffs, int s_max) {
    if (num_rows < 1 || num_heads < 1 || num_heads > SMLA_MAX_HEADS || kv_len < 0 ||
        s_max < 1 || s_max > SMLA_MAX_SPLITS)
        return -(int)SMLA_ERR_BAD_SHAPE;
    const smla_plan_coeffs& c = coeffs != nullptr ? *coeffs : kGB300Coeffs;
    if (!(c.slots >= 1.0)) return -(int)SMLA_ERR_BAD_SHAPE;
    const int64_t slots = (int64_t)c.slots;
    int best_s = 1;
    double best = 0.0;
    for (int s = 1; s <= s_max; ++s) {
        const int64_t units = (int64_t)num_rows * s;
        const double waves = (double)((units + slots - 1) / slots);
        const double per_wave = c.t0 + c.c_entry * (double)((kv_len + s - 1) / s);
        double cost = waves * per_wave;
        if (s > 1) cost += c.c_byte * (double)((int64_t)num_rows * num_heads * SMLA_HEAD_DIM * 4 * s) + c.c_merge;
        if (s == 1 || cost < best) {
            best = cost;
            best_s = s;
        }
    }
    return best_s;
}

int smla_plan_num_splits(int num_rows, int num_heads, int64_t kv_len) {
    return smla_plan_num_splits_ex(num_rows, num_heads, kv_len, nullptr, SMLA_MAX_SPLITS);
}

size_t smla_workspace_bytes(int max_rows, int num_heads, int max_splits) {
    if (max_rows < 1 || max_rows > SMLA_MAX_ROWS || num_heads < 1 || num_heads > SMLA_MAX_HEADS ||
        max_splits < 1 || max_splits > SMLA_MAX_SPLITS)
        return 0;
    return smla::workspace_layout(max_rows, num_heads, max_splits).total;
}

smla_status smla_decode(const smla_decode_args* a, void* workspace, size_t ws_bytes, smla_stream_t stream) {
    const smla_status st = smla::check_decode_call(a, workspace, ws_bytes);
    if (st != SMLA_OK) return st;
    return smla::launch_decode(a, workspace, static_cast<cudaStream_t>(stream));
}

smla_status smla_read_device_error(void* workspace, uint32_t* flags, smla_stream_t stream) {
    if (workspace == nullptr || flags == nullptr) return SMLA_ERR_NULL_POINTER;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SMLA_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return SMLA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SMLA_ERR_CUDA;
    *flags = host;
    return SMLA_OK;
}

uint64_t smla_set_wait_limit_ns(uint64_t ns) {
    return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

const char* smla_status_string(smla_status status) {
    switch (status) {
        case SMLA_OK: return "ok";
        case SMLA_ERR_NULL_POINTER: return "a required pointer is NULL";
        case SMLA_ERR_MISALIGNED: return "a pointer breaks its required alignment";
        case SMLA_ERR_BAD_SHAPE: return "a size argument is out of range";
        case SMLA_ERR_WORKSPACE_TOO_SMALL: return "workspace is smaller than smla_workspace_bytes()";
        case SMLA_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103 (GB300)";
        case SMLA_ERR_CUDA: return "CUDA runtime error or launch failure";
    }
    return "unknown status";
}

}  // extern "C"
