// Top-k selection: per row, the k positions of [0, len_r) with the largest
// scores -- the decode's top-k index list (-1 = invalid slot).
//
// The pages name this producer (the indexer top-k path whose cp-gather is
// reworked in "[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on
// gfx950", comment "8k/1k TP8 follow-up", item 2) but not how the scores are
// made, so the scores are an input.  Order: score descending, ties by position
// ascending; NaN scores are never selected; a row with fewer than k
// selectable positions is padded with -1.
//
// One CTA per row.  Scores map to order-preserving 32-bit keys (NaN -> 0, the
// one key never selected).  A radix select over the key's 11 + 11 + 10 bits
// (histograms in shared memory) finds the k-th largest key T; one more pass
// collects every key above T and, in position order, the first positions
// equal to T; a bitonic sort in shared memory orders the k results.
#include <cstdint>
#include <cuda_runtime.h>

#include "smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kThreadsTopk = 1024;
constexpr int kMaxK = SMLA_TOPK_MAX_K;

// Order-preserving key: a larger score gives a larger key; -0 and +0 are one
// key (they compare equal); NaN gives 0, the one key never selected.
__device__ __forceinline__ uint32_t sort_key(float f) {
    if (f != f) return 0u;
    const uint32_t b = f == 0.f ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kThreadsTopk) smla_topk_kernel(const float* __restrict__ scores, int64_t stride,
                                                                 const int32_t* __restrict__ lens, int k,
                                                                 int32_t* __restrict__ out) {
    __shared__ uint32_t hist[2048];
    __shared__ unsigned long long sel[kMaxK];  // (key << 32) | ~position: larger = earlier in the output
    __shared__ uint32_t s_prefix, s_mask, s_need, s_count, s_gt;
    __shared__ uint32_t s_warp[kThreadsTopk / 32];
    const int r = blockIdx.x, tid = threadIdx.x;
    const float* row = scores + (int64_t)r * stride;
    const int L = (int)min((int64_t)max(0, __ldg(lens + r)), stride);  // lengths past the row's capacity are cut
    const bool vec4 = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;    // 16-byte loads where the row allows
    // ---- radix select: the k-th largest key among keys >= 1
    if (tid == 0) { s_prefix = 0u; s_mask = 0u; s_need = (uint32_t)k; }
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    uint32_t total_valid = 0;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass], nb = 1 << widths[pass];
        for (int i = tid; i < nb; i += kThreadsTopk) hist[i] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        auto count = [&](float f) {
            const uint32_t key = sort_key(f);
            if (key != 0u && (key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (uint32_t)(nb - 1)], 1u);
        };
        if (vec4) {
            const float4* row4 = reinterpret_cast<const float4*>(row);
            for (int i = tid; i < L / 4; i += kThreadsTopk) {
                const float4 v = __ldg(row4 + i);
                count(v.x); count(v.y); count(v.z); count(v.w);
            }
            for (int i = (L & ~3) + tid; i < L; i += kThreadsTopk) count(__ldg(row + i));
        } else {
            for (int i = tid; i < L; i += kThreadsTopk) count(__ldg(row + i));
        }
        __syncthreads();
        if (tid == 0) {  // walk the bins from the top until the k-th key's bin
            uint32_t need = s_need, acc = 0;
            int b = nb - 1;
            if (pass == 0) {
                uint32_t tot = 0;
                for (int j = 0; j < nb; ++j) tot += hist[j];
                s_count = tot;  // valid keys in the row
            }
            for (; b > 0; --b) {
                if (acc + hist[b] >= need) break;
                acc += hist[b];
            }
            s_need = need - acc;  // still needed from bin b
            s_prefix = prefix | ((uint32_t)b << sh);
            s_mask = mask | ((uint32_t)(nb - 1) << sh);
        }
        __syncthreads();
        if (pass == 0) total_valid = s_count;
    }
    // T = s_prefix; every key > T is taken, and s_need keys equal to T (the
    // smallest positions).  With fewer valid keys than k, take them all.
    const bool take_all = total_valid <= (uint32_t)k;
    const uint32_t T = take_all ? 1u : s_prefix;
    const uint32_t need_eq = take_all ? 0xFFFFFFFFu : s_need;
    const int n_sel = take_all ? (int)total_valid : k;
    if (tid == 0) { s_count = 0u; s_gt = 0u; }
    __syncthreads();
    // ---- collect: keys above T anywhere; keys equal to T in position order
    uint32_t eq_base = 0;  // equal keys taken by earlier chunks
    for (int base = 0; base < L; base += kThreadsTopk) {
        const int i = base + tid;
        const uint32_t key = i < L ? sort_key(__ldg(row + i)) : 0u;
        const unsigned long long item = ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)i;
        if (key > T || (take_all && key != 0u)) {
            const uint32_t slot = atomicAdd(&s_count, 1u);
            sel[slot] = item;
        }
        if (!take_all) {  // equal keys: taken in position order until need_eq
            const bool eq = key == T && key != 0u;
            const uint32_t chunk_total = (uint32_t)__syncthreads_count(eq);
            if (chunk_total != 0u && eq_base < need_eq) {  // block-uniform: the rare chunks holding T
                const uint32_t ballot = __ballot_sync(0xffffffffu, eq);
                if ((tid & 31) == 0) s_warp[tid >> 5] = __popc(ballot);
                __syncthreads();
                uint32_t before = eq_base;
                for (int w = 0; w < (tid >> 5); ++w) before += s_warp[w];
                before += __popc(ballot & ((1u << (tid & 31)) - 1u));
                if (eq && before < need_eq) {
                    const uint32_t slot = atomicAdd(&s_count, 1u);
                    sel[slot] = item;
                }
                __syncthreads();
            }
            eq_base += chunk_total;
        }
    }
    __syncthreads();
    // ---- bitonic sort of the selected items, descending (pad with 0)
    int n2 = 1;
    while (n2 < n_sel) n2 <<= 1;
    for (int i = n_sel + tid; i < n2; i += kThreadsTopk) sel[i] = 0ull;
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride2 = size >> 1; stride2 > 0; stride2 >>= 1) {
            for (int i = tid; i < n2; i += kThreadsTopk) {
                const int j = i ^ stride2;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long a = sel[i], b = sel[j];
                    if (desc ? (a < b) : (a > b)) { sel[i] = b; sel[j] = a; }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < k; i += kThreadsTopk)
        out[(int64_t)r * k + i] = i < n_sel ? (int32_t)~(uint32_t)(sel[i] & 0xFFFFFFFFull) : -1;
}

}  // namespace
}  // namespace smla

extern "C" smla_status smla_topk_indices(const float* scores, int64_t stride, const int32_t* lens, int32_t num_rows,
                                         int32_t k, int32_t* out, smla_stream_t stream) {
    using namespace smla;
    if (num_rows < 0 || k < 1 || k > SMLA_TOPK_MAX_K || stride < 0 || stride > INT32_MAX) return SMLA_ERR_BAD_SHAPE;
    if (num_rows == 0) return SMLA_OK;
    if (scores == nullptr || lens == nullptr || out == nullptr) return SMLA_ERR_NULL_POINTER;
    if ((reinterpret_cast<uintptr_t>(scores) & 3u) || (reinterpret_cast<uintptr_t>(lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(out) & 3u))
        return SMLA_ERR_MISALIGNED;
    const smla_status dev = check_device_only();
    if (dev != SMLA_OK) return dev;
    smla_topk_kernel<<<num_rows, kThreadsTopk, 0, static_cast<cudaStream_t>(stream)>>>(scores, stride, lens, k, out);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}
