// Top-k selection: per row, the k positions of [0, len_r) with the largest
// scores -- the decode's top-k index list (-1 = invalid slot).
//
// The cited page names this producer (the indexer top-k path whose cp-gather
// is reworked in "[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on
// gfx950", comment "8k/1k TP8 follow-up", item 2) but not how the scores are
// made, so the scores are an input.  Order: score descending, ties by position
// ascending; NaN scores are never selected; a row with fewer than k
// selectable positions is padded with -1.
//
// A cluster of two CTAs per row, each over a contiguous half of it; their
// histograms are summed through distributed shared memory and every selected
// key lands in the first CTA's buffer.  Scores map to order-preserving 32-bit
// keys (NaN -> 0, the one key never selected).
//
// Usually one read of the row: a sample (the first 64 scores of every 1024)
// places a 24-bit key prefix tau that about 1.45 k keys reach; the first pass
// collects every key whose prefix is >= tau (one float comparison per score).
// When that collected between k and SMLA_TOPK_MAX_K keys (or, with tau = 0,
// every valid key), they hold the top k.  Otherwise a radix select runs over
// the row (13 + 11 + 8 key
// bits, the bin of the k-th largest key found by a block-wide suffix scan): as
// soon as the keys at or above the
// current bin number at most SMLA_TOPK_MAX_K, one more pass collects exactly
// those; with many keys tied at the threshold, the third pass gives the k-th
// largest key T and a collecting pass takes every key above T and, in
// position order (the second half's ties after the first's), the first
// positions equal to T.  The selected keys are sorted (key descending,
// position ascending) by a bitonic network over the block: registers and
// shuffles within a warp, shared memory across warps.
#include <atomic>
#include <cstdint>
#include <mutex>
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreadsTopk = 1024;
constexpr int kMaxK = SMLA_TOPK_MAX_K;
constexpr int kMaxBins = 1 << 13;  // the first pass's histogram
constexpr int kGuessNum = 29, kGuessDen = 20;  // kGuessFactor = 1.45: the guess aims at 1.45 k keys
constexpr int kMaxTies = 1024;   // ties at the k-th key ranked directly (more: all collected keys sorted)
constexpr int kCluster = 2;        // CTAs per row (a thread-block cluster), each over a contiguous part
constexpr size_t kTopkSmem = kMaxK * 8 + 2 * kMaxBins * 4;  // selection + part and cluster histograms

// Order-preserving key: a larger score gives a larger key; -0 and +0 are one
// key (they compare equal); NaN gives 0, the one key never selected.
__device__ __forceinline__ uint32_t sort_key(float f) {
    if (f != f) return 0u;
    const uint32_t b = f == 0.f ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // sort_key(-inf): every key below it is a NaN's bit pattern

// The float whose key is `key` (key >= kKeyNegInf): for a score f that is not
// NaN, sort_key(f) >= key exactly when f >= key_float(key) (the keys follow
// the float order, and -0 >= +0 as their shared key requires); a NaN fails
// the comparison, as its key 0 would.
__device__ __forceinline__ float key_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Calls f(score, position) for every position of [0, L) of `row`: 16-byte
// loads where the row is 16-byte aligned, eight of them in flight per thread.
template <class F>
__device__ __forceinline__ void for_each_score(const float* __restrict__ row, int L, bool vec4, F f) {
    const int tid = threadIdx.x;
    if (vec4) {
        const float4* row4 = reinterpret_cast<const float4*>(row);
        const int n4 = L / 4;
        int i = tid;
        for (; i + 7 * kThreadsTopk < n4; i += 8 * kThreadsTopk) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldg(row4 + i + u * kThreadsTopk);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int b = 4 * (i + u * kThreadsTopk);
                f(v[u].x, b); f(v[u].y, b + 1); f(v[u].z, b + 2); f(v[u].w, b + 3);
            }
        }
        for (; i < n4; i += kThreadsTopk) {
            const float4 v = __ldg(row4 + i);
            f(v.x, 4 * i); f(v.y, 4 * i + 1); f(v.z, 4 * i + 2); f(v.w, 4 * i + 3);
        }
        for (int j = (L & ~3) + tid; j < L; j += kThreadsTopk) f(__ldg(row + j), j);
    } else {
        for (int j = tid; j < L; j += kThreadsTopk) f(__ldg(row + j), j);
    }
}

// The bin b of hist[0, nb) holding the need-th largest key (need >= 1): the
// largest b with sum_{j >= b} hist[j] >= need, and acc = sum_{j > b} hist[j];
// b = 0 when the bins hold fewer than need keys.  Thread t sums bins
// [t per, (t + 1) per); a block suffix scan of those sums points one thread at
// the crossing, which walks its own bins.  Written by that thread into *b_out
// and *acc_out; the total into *tot_out (thread 0) unless it is null.  All
// threads call it.
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, uint32_t need, uint32_t* s_warp,
                                         uint32_t* b_out, uint32_t* acc_out, uint32_t* tot_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = max(1, nb / kThreadsTopk);
    const int lo = tid * per, hi = min(nb, lo + per);
    uint32_t sum = 0;
    for (int b = lo; b < hi; ++b) sum += hist[b];
    // inclusive suffix sum over the warp's lanes (lanes above this one, and it)
    uint32_t suf = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += v;
    }
    if (lane == 0) s_warp[warp] = suf;  // the warp's total
    __syncthreads();
    uint32_t above = suf - sum;  // lanes above in this warp
    for (int w = warp + 1; w < kThreadsTopk / 32; ++w) above += s_warp[w];
    const uint32_t total_here = above + sum;
    const bool mine = (above < need && need <= total_here) || (tid == 0 && total_here < need);
    if (mine) {
        uint32_t acc = above;
        int b = hi - 1;
        for (; b > lo; --b) {
            if (acc + hist[b] >= need) break;
            acc += hist[b];
        }
        *b_out = (uint32_t)b;
        *acc_out = acc;
    }
    if (tid == 0 && tot_out != nullptr) *tot_out = total_here;
    __syncthreads();
}

__device__ __forceinline__ unsigned long long sel_item(uint32_t key, int pos) {
    return ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)pos;  // larger = earlier in the output
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreadsTopk)
    smla_topk_kernel(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ lens, int k,
                     int32_t* __restrict__ out) {
    extern __shared__ unsigned long long topk_smem[];
    unsigned long long* sel = topk_smem;                                         // [kMaxK] (rank 0 gathers)
    uint32_t* hist = reinterpret_cast<uint32_t*>(topk_smem + kMaxK);              // [kMaxBins] this CTA's part
    uint32_t* comb = hist + kMaxBins;                                             // [kMaxBins] the cluster's sum
    __shared__ uint32_t s_prefix, s_mask, s_need, s_count, s_total, s_bin, s_b, s_acc, s_sampled;
    __shared__ uint32_t s_warp[kThreadsTopk / 32];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int r = blockIdx.x / kCluster, tid = threadIdx.x;
    const float* row = scores + (int64_t)r * stride;
    const int L = (int)min((int64_t)max(0, __ldg(lens + r)), stride);  // lengths past the row's capacity are cut
    const bool vec4 = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;    // 16-byte loads where the row allows
    // this CTA's contiguous part of the row (a multiple of 4 positions long)
    const int seg = ((L + kCluster - 1) / kCluster + 3) & ~3;
    const int beg = min(L, rank * seg), end = min(L, beg + seg);
    const float* part = row + beg;
    // rank 0's counter and selection buffer, which every CTA of the cluster fills
    uint32_t* cnt0 = cl.map_shared_rank(&s_count, 0);
    unsigned long long* sel0 = cl.map_shared_rank(sel, 0);
    if (tid == 0) { s_prefix = 0u; s_mask = 0u; s_need = (uint32_t)k; s_count = 0u; }
    const int shifts[3] = {19, 8, 0};
    const int widths[3] = {13, 11, 8};
    bool fast = false;
    // ---- a guess of the threshold from a sample of each part (the first 64
    // scores of every 1024: contiguous runs, so that DRAM bursts are not
    // wasted): the 24-bit key prefix tau whose keys and those above
    // it number about kGuessFactor k in the sample, scaled to the row; found
    // by a 13-bit histogram of the sample and then an 11-bit one of the sampled
    // keys in the chosen bin (a second read of the sample, from L2).  The first
    // pass then collects the keys whose prefix is >= tau.
    uint32_t guess = 0xFFFFFFFFu;  // no guess: nothing is collected in the first pass
    {
        const int plen = end - beg;
        // sampled float4s (or scores): j -> run j / 16 (64), item j % 16 (64)
        const int ns = vec4 ? 16 * ((plen / 4) / 256) + min(16, (plen / 4) % 256)
                            : 64 * (plen / 1024) + min(64, plen % 1024);
        // f(key) for every sampled key, eight loads in flight per thread
        auto for_each_sample = [&](auto f) {
            if (vec4) {
                const float4* p4 = reinterpret_cast<const float4*>(part);
                int j = tid;
                for (; j + 7 * kThreadsTopk < ns; j += 8 * kThreadsTopk) {
                    float4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int jj = j + u * kThreadsTopk;
                        v[u] = __ldg(p4 + (size_t)(jj >> 4) * 256 + (jj & 15));
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) { f(sort_key(v[u].x)); f(sort_key(v[u].y)); f(sort_key(v[u].z)); f(sort_key(v[u].w)); }
                }
                for (; j < ns; j += kThreadsTopk) {
                    const float4 v = __ldg(p4 + (size_t)(j >> 4) * 256 + (j & 15));
                    f(sort_key(v.x)); f(sort_key(v.y)); f(sort_key(v.z)); f(sort_key(v.w));
                }
            } else {
                for (int j = tid; j < ns; j += kThreadsTopk) f(sort_key(__ldg(part + (size_t)(j >> 6) * 1024 + (j & 63))));
            }
        };
        for (int i = tid; i < kMaxBins; i += kThreadsTopk) hist[i] = 0u;
        if (tid == 0) s_sampled = (uint32_t)(vec4 ? 4 * ns : ns);
        __syncthreads();
        for_each_sample([&](uint32_t key) { if (key != 0u) atomicAdd(&hist[key >> 19], 1u); });
        cl.sync();  // every part's sample histogram and size are complete
        uint32_t sampled = 0;
        for (int q = 0; q < kCluster; ++q) sampled += *cl.map_shared_rank(&s_sampled, q);
        for (int i = tid; i < kMaxBins; i += kThreadsTopk) {
            uint32_t v = 0;
#pragma unroll
            for (int q = 0; q < kCluster; ++q) v += cl.map_shared_rank(hist, q)[i];
            comb[i] = v;
        }
        __syncthreads();
        // the sample's share of kGuessFactor k, at least one key
        const uint32_t want = (uint32_t)max(
            1ll, ((long long)kGuessNum * k * sampled + (long long)kGuessDen * max(L, 1) - 1) /
                     ((long long)kGuessDen * max(L, 1)));
        find_bin(comb, kMaxBins, want, s_warp, &s_b, &s_acc, &s_total);
        const uint32_t b1 = s_b, need1 = want - s_acc, tot = s_total;
        cl.sync();  // the other parts have read this histogram before it is cleared
        if (tot >= want) {  // uniform: enough valid sample keys to place tau
            for (int i = tid; i < 2048; i += kThreadsTopk) hist[i] = 0u;
            __syncthreads();
            for_each_sample([&](uint32_t key) {
                if (key != 0u && (key >> 19) == b1) atomicAdd(&hist[(key >> 8) & 0x7FFu], 1u);
            });
            cl.sync();
            for (int i = tid; i < 2048; i += kThreadsTopk) {
                uint32_t v = 0;
#pragma unroll
                for (int q = 0; q < kCluster; ++q) v += cl.map_shared_rank(hist, q)[i];
                comb[i] = v;
            }
            __syncthreads();
            find_bin(comb, 2048, need1, s_warp, &s_b, &s_acc, nullptr);
            guess = (b1 << 11) | s_b;  // tau: the top 24 bits
            cl.sync();  // the other parts have read this histogram before it is cleared
        } else {
            guess = 0u;  // the sample holds fewer valid keys than wanted: collect every valid key
        }
    }
    if (guess != 0xFFFFFFFFu) {
        // collect the valid keys whose prefix is >= tau: the scores >= the float
        // of key max(tau << 8, the key of -inf) (tau = 0: every valid key)
        const float fthr = key_float(max(guess << 8, kKeyNegInf));
        for_each_score(part, end - beg, vec4, [&](float f, int i) {
            if (f >= fthr) {
                const uint32_t slot = atomicAdd(cnt0, 1u);
                if (slot < (uint32_t)kMaxK) sel0[slot] = sel_item(sort_key(f), beg + i);
            }
        });
        cl.sync();  // every part's keys are in (rank 0's counter is settled)
        // the guess held if it collected between k and kMaxK keys, or with tau = 0
        // every valid key, at most kMaxK (rank 0's counter keeps counting past
        // kMaxK); a row with fewer than k valid keys at a tau above 0 takes the
        // radix select
        const uint32_t n_spec = *cnt0;
        if ((n_spec >= (uint32_t)k || guess == 0u) && n_spec <= (uint32_t)kMaxK) {
            fast = true;
        } else {
            cl.sync();  // every part has read the counter
            // a miss: rank 0's buffer is emptied before anything is collected again
            if (tid == 0) s_count = 0u;
            cl.sync();
        }
    }
#pragma unroll 1
    for (int pass = 0; pass < 3 && !fast; ++pass) {
        const int sh = shifts[pass], nb = 1 << widths[pass];
        for (int i = tid; i < nb; i += kThreadsTopk) hist[i] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        for_each_score(part, end - beg, vec4, [&](float f, int) {
            const uint32_t key = sort_key(f);
            if (key != 0u && (key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (uint32_t)(nb - 1)], 1u);
        });
        cl.sync();  // every part's histogram is complete
        for (int i = tid; i < nb; i += kThreadsTopk) {
            uint32_t v = 0;
#pragma unroll
            for (int q = 0; q < kCluster; ++q) v += cl.map_shared_rank(hist, q)[i];
            comb[i] = v;
        }
        __syncthreads();
        const uint32_t need = s_need;
        find_bin(comb, nb, need, s_warp, &s_b, &s_acc, pass == 0 ? &s_total : nullptr);
        if (tid == 0) {
            const uint32_t b = s_b;
            s_need = need - s_acc;  // still needed from bin b
            s_bin = comb[b];
            s_prefix = prefix | (b << sh);
            s_mask = mask | ((uint32_t)(nb - 1) << sh);
        }
        __syncthreads();
        // keys at or above the bin: k - need above it, plus the bin's own
        const uint32_t at_or_above = (uint32_t)k - s_need + s_bin;
        const bool all_fit = pass == 0 && s_total <= (uint32_t)kMaxK;
        if (all_fit || at_or_above <= (uint32_t)kMaxK) {
            // one pass collects them, unordered, into rank 0's buffer
            const uint32_t cp = all_fit ? 0u : s_prefix, cm = all_fit ? 0u : s_mask;
            for_each_score(part, end - beg, vec4, [&](float f, int i) {
                const uint32_t key = sort_key(f);
                if (key != 0u && (key & cm) >= cp) {
                    const uint32_t slot = atomicAdd(cnt0, 1u);
                    if (slot < (uint32_t)kMaxK) sel0[slot] = sel_item(key, beg + i);
                }
            });
            fast = true;
            break;
        }
        if (pass < 2) cl.sync();  // the other parts have read this histogram before it is cleared
    }
    if (!fast) {
        // Many keys tied at the threshold: T = s_prefix is the k-th largest key;
        // every key > T is taken, and s_need keys equal to T (the smallest
        // positions), collected in position order: this part's ties follow
        // those of the parts before it, counted by their last histograms.
        const uint32_t T = s_prefix, need_eq = s_need, bT = T & 0xFFu;
        uint32_t eq_base = 0;  // equal keys taken before this part's current chunk
        for (int q = 0; q < rank; ++q) eq_base += cl.map_shared_rank(hist, q)[bT];
        for (int base = beg; base < end; base += kThreadsTopk) {
            const int i = base + tid;
            const uint32_t key = i < end ? sort_key(__ldg(row + i)) : 0u;
            if (key > T) {
                const uint32_t slot = atomicAdd(cnt0, 1u);
                sel0[slot] = sel_item(key, i);
            }
            const bool eq = key == T && key != 0u;
            const uint32_t chunk_total = (uint32_t)__syncthreads_count(eq);
            if (chunk_total != 0u && eq_base < need_eq) {  // block-uniform: the chunks holding T
                const uint32_t ballot = __ballot_sync(0xffffffffu, eq);
                if ((tid & 31) == 0) s_warp[tid >> 5] = __popc(ballot);
                __syncthreads();
                uint32_t before = eq_base;
                for (int w = 0; w < (tid >> 5); ++w) before += s_warp[w];
                before += __popc(ballot & ((1u << (tid & 31)) - 1u));
                if (eq && before < need_eq) {
                    const uint32_t slot = atomicAdd(cnt0, 1u);
                    sel0[slot] = sel_item(key, i);
                }
                __syncthreads();
            }
            eq_base += chunk_total;
        }
    }
    cl.sync();  // every part's keys sit in rank 0's buffer; no CTA reads another's memory after this
    if (rank != 0) return;
    int n_sel = fast ? (int)min(s_count, (uint32_t)kMaxK) : k;
    // ---- more than k collected: keep exactly the top k.  A radix select over
    // the collected keys (11 + 11 + 10 bits, histograms in shared memory) gives
    // the k-th largest key T; every key above T stays, and of the keys equal to
    // T the need_eq with the smallest positions (each tie's rank among the ties
    // counted directly; with more than kMaxTies ties all are sorted instead).
    unsigned long long* kept = reinterpret_cast<unsigned long long*>(comb);  // [kMaxK / 2 ...]: 32 KB
    if (n_sel > k) {
        uint32_t prefix = 0u, mask = 0u, need = (uint32_t)k, count_t = 0u;
        const int shs[3] = {21, 10, 0}, wds[3] = {11, 11, 10};
#pragma unroll 1
        for (int lvl = 0; lvl < 3; ++lvl) {
            const int sh = shs[lvl], nb = 1 << wds[lvl];
            for (int i = tid; i < nb; i += kThreadsTopk) hist[i] = 0u;
            __syncthreads();
            for (int i = tid; i < n_sel; i += kThreadsTopk) {
                const uint32_t key = (uint32_t)(sel[i] >> 32);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (uint32_t)(nb - 1)], 1u);
            }
            __syncthreads();
            find_bin(hist, nb, need, s_warp, &s_b, &s_acc, nullptr);
            const uint32_t b = s_b;
            need -= s_acc;
            count_t = hist[b];
            prefix |= b << sh;
            mask |= (uint32_t)(nb - 1) << sh;
            __syncthreads();  // hist read before the next level clears it
        }
        const uint32_t T = prefix, need_eq = need;  // 1 <= need_eq <= count_t
        if (count_t == need_eq || count_t <= (uint32_t)kMaxTies) {
            unsigned long long* ties = reinterpret_cast<unsigned long long*>(hist);  // [kMaxTies]
            if (tid == 0) { s_count = 0u; s_acc = 0u; }
            __syncthreads();
            for (int i = tid; i < n_sel; i += kThreadsTopk) {
                const unsigned long long it = sel[i];
                const uint32_t key = (uint32_t)(it >> 32);
                if (key > T || (key == T && count_t == need_eq)) kept[atomicAdd(&s_count, 1u)] = it;
                else if (key == T) ties[atomicAdd(&s_acc, 1u)] = it;
            }
            __syncthreads();
            if (count_t != need_eq) {  // the need_eq ties with the largest items (smallest positions)
                const int nt = (int)s_acc;
                for (int i = tid; i < nt; i += kThreadsTopk) {
                    const unsigned long long it = ties[i];
                    int rank = 0;
                    for (int j = 0; j < nt; ++j) rank += ties[j] > it;
                    if (rank < (int)need_eq) kept[atomicAdd(&s_count, 1u)] = it;
                }
                __syncthreads();
            }
            for (int i = tid; i < k; i += kThreadsTopk) sel[i] = kept[i];
            __syncthreads();
            n_sel = k;
        }
    }
    // ---- sort of the n_sel items, descending (padded with 0 to n2, a power of
    // two from 128 to kMaxK): a bitonic network over the block.  Thread t holds
    // items 4t .. 4t + 3 in registers; compare-exchange steps of stride 1 and 2
    // pair items of one thread, strides 4 .. 64 items of one warp (through
    // shuffles), and strides of 128 and more items of other warps, through
    // shared memory (two buffers used in turn, so one barrier per step: a
    // buffer is written again only after the step between has made every
    // thread finish reading it).  Threads past n2 / 4 hold nothing (whole
    // warps, as n2 >= 128).
    static_assert(kMaxK == 4 * kThreadsTopk, "four items per thread");
    int n2 = 128;
    while (n2 < n_sel) n2 <<= 1;
    const bool holds = 4 * tid < n2;
    for (int i = n_sel + tid; i < n2; i += kThreadsTopk) sel[i] = 0ull;
    __syncthreads();
    unsigned long long x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = holds ? sel[4 * tid + u] : 0ull;
    unsigned long long* const buf1 = reinterpret_cast<unsigned long long*>(hist);  // hist + comb: idle now
    bool cur = false;
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride2 = size >> 1; stride2 > 0; stride2 >>= 1) {
            if (stride2 >= 128) {  // partners in other warps (block-uniform branch)
                unsigned long long* const b = cur ? buf1 : sel;
                if (holds) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) b[4 * tid + u] = x[u];
                }
                __syncthreads();
                if (holds) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = 4 * tid + u, j = i ^ stride2;
                        const unsigned long long y = b[j];
                        const bool desc = (i & size) == 0, lower = i < j;
                        x[u] = (desc == lower) ? (x[u] > y ? x[u] : y) : (x[u] < y ? x[u] : y);
                    }
                }
                cur = !cur;
            } else if (holds) {
                if (stride2 >= 4) {  // partners in this warp: lane ^ (stride2 / 4)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = 4 * tid + u, j = i ^ stride2;
                        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x[u], stride2 >> 2);
                        const bool desc = (i & size) == 0, lower = i < j;
                        x[u] = (desc == lower) ? (x[u] > y ? x[u] : y) : (x[u] < y ? x[u] : y);
                    }
                } else {  // partners in this thread: (0, 2), (1, 3) for stride 2; (0, 1), (2, 3) for stride 1
                    auto cx = [&](unsigned long long& a, unsigned long long& b, int i) {  // i: a's index
                        const bool desc = (i & size) == 0;
                        if (desc ? (a < b) : (a > b)) { const unsigned long long t = a; a = b; b = t; }
                    };
                    if (stride2 == 2) { cx(x[0], x[2], 4 * tid); cx(x[1], x[3], 4 * tid + 1); }
                    else { cx(x[0], x[1], 4 * tid); cx(x[2], x[3], 4 * tid + 2); }
                }
            }
        }
    }
    // the sorted items straight from registers: item i -> out[i]
    const int n_out = min(n_sel, k);
    if (holds) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = 4 * tid + u;
            if (i < k) out[(int64_t)r * k + i] = i < n_out ? (int32_t)~(uint32_t)(x[u] & 0xFFFFFFFFull) : -1;
        }
    }
    for (int i = n2 + tid; i < k; i += kThreadsTopk) out[(int64_t)r * k + i] = -1;
}

std::atomic<int> g_topk_attr[64];
std::mutex g_topk_mu;

// The kernel takes more than 48 KB of dynamic shared memory: opt in once per device.
cudaError_t ensure_topk_attrs() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_topk_attr[dev].load(std::memory_order_acquire) == 1) return cudaSuccess;
    std::lock_guard<std::mutex> lk(g_topk_mu);
    if (g_topk_attr[dev].load(std::memory_order_relaxed) == 1) return cudaSuccess;
    e = cudaFuncSetAttribute(smla_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTopkSmem);
    if (e != cudaSuccess) return e;
    g_topk_attr[dev].store(1, std::memory_order_release);
    return cudaSuccess;
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
    if (ensure_topk_attrs() != cudaSuccess) return SMLA_ERR_CUDA;
    smla_topk_kernel<<<num_rows * kCluster, kThreadsTopk, kTopkSmem, static_cast<cudaStream_t>(stream)>>>(scores, stride, lens, k,
                                                                                                out);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}
