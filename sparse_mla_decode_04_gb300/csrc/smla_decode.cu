// Sparse-MLA decode for sm_103a: kernel and launch.
//
// Method ("[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on gfx950",
// section "Design"): per query row, one 512-wide QK dot (448 NoPE + 64 RoPE
// dims) against the entries the row selects (top-k main-cache slots with -1 as
// an invalid slot, a sliding window, compressed-cache 64-entry groups with a
// masked tail), a softmax with a per-head sink logit, and a 512-wide PV.
// Split plan, last-arriver merge and graph safety follow "[ASM] [HIP] [MLA v4
// nm] Split plan helper and persistent decode kernel with in-kernel split and
// merge", summary part 2.
//
// GB300 design.  A work unit is (row, split).  Each unit runs on a CTA pair
// (cluster of 2); CTA c owns dims [256c, 256c+256) of the 512-wide head dim:
//   * it gathers and dequantises only its half of every entry (fp8 e4m3 x
//     UE8M0 -> bf16, exact) into a 128-byte-swizzled shared-memory tile that
//     serves as the K-major B operand of QK and the MN-major B operand of PV;
//   * QK over its 256 dims runs on tcgen05 (M = 128 heads, N = 64 entries,
//     K = 256) into TMEM; the two partial score tiles are exchanged through
//     distributed shared memory and summed (fp32 addition commutes, so both
//     CTAs hold bit-identical scores and take identical softmax decisions);
//   * P goes to shared memory as two bf16 tiles, hi = bf16(p) and
//     lo = bf16(p - hi), and PV (M = 128, N = 256, K = 64) runs once per tile
//     of the pair, accumulating into this CTA's 256 TMEM columns of O.  A
//     single bf16 P (8-bit mantissa) is not enough here: with V up to ~600 in
//     magnitude, two nearly tied entries whose V values cancel would carry
//     errors near 1, while hi + lo carries p to ~2^-17.
// TMEM per CTA: O 256 columns + S 64 columns (512 allocated).
// Heads beyond num_heads are zero-padded up to the MMA's M = 128.
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "smla.h"
#include "smla_internal.h"
#include "sm103_ptx.cuh"

namespace smla {

constexpr int kBK = 64;            // entries per tile
constexpr int kThreads = 128;      // one thread per (padded) head
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;   // partial S: columns [256, 320)
constexpr uint64_t kWaitNs = 2000000000ull;  // bounded-wait limit (2 s)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Shared-memory layout (offsets from a 1024-byte-aligned base).
constexpr uint32_t kOffQ = 0;                      // [4 atoms][128 heads][128 B]   64 KB
constexpr uint32_t kOffX = kOffQ + 65536;          // [4 atoms][64 entries][128 B]  32 KB
constexpr uint32_t kOffP = kOffX + 32768;          // P hi part [128 heads][128 B]  16 KB
constexpr uint32_t kOffPlo = kOffP + 16384;        // P lo part [128 heads][128 B]  16 KB
constexpr uint32_t kOffSin = kOffPlo + 16384;      // peer's partial S [128][64] f32 32 KB
constexpr uint32_t kOffSlotE = kOffSin + 32768;    // entry pointers [64]
constexpr uint32_t kOffSlotS = kOffSlotE + 512;    // scale pointers [64]
constexpr uint32_t kOffTiles = kOffSlotS + 512;    // int32 tiles per row [kMaxRows]
constexpr uint32_t kOffPrefix = kOffTiles + 4 * SMLA_MAX_ROWS;          // int32 [kMaxRows + 1]
constexpr uint32_t kOffBar = kOffPrefix + 4 * (SMLA_MAX_ROWS + 8);     // mbarriers
constexpr uint32_t kOffMisc = kOffBar + 64;        // tmem base, flags, reduction scratch
constexpr uint32_t kSmemUsed = kOffMisc + 256;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack

struct KParams {
    smla_decode_args a;
    uint32_t* err;
    uint32_t* counters;  // [SMLA_MAX_ROWS][2]
    float2* ml;          // [units][2][H]   (m in log2 units, l)
    float* po;           // [units][H][512] unnormalised fp32 O
    int units;           // num_rows * num_splits
};

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ float ue8m0_to_f32(uint32_t code) {
    if (code == 0u) return __uint_as_float(0x00400000u);   // 2^-127 (subnormal)
    if (code == 255u) return __uint_as_float(0x7fffffffu); // NaN
    return __uint_as_float(code << 23);                    // 2^(code-127)
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &b, 4);
    return u;
}

// 16 fp8-e4m3 codes * scale -> 16 bf16 (8 packed words).  Exact: an e4m3
// value times a power of two is representable in bf16 when the product is a
// bf16 normal.
__device__ __forceinline__ void dequant16(const uint4 raw, float scale, uint32_t (&o)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i] >> (16 * j)) & 0xFFFFu);
            const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            __half lo, hi;
            memcpy(&lo, &h2.x, 2);
            memcpy(&hi, &h2.y, 2);
            const float flo = __half2float(lo) * scale;
            const float fhi = __half2float(hi) * scale;
            const __nv_bfloat162 b = __floats2bfloat162_rn(flo, fhi);
            uint32_t u;
            memcpy(&u, &b, 4);
            o[2 * i + j] = u;
        }
    }
}

// (a, b) -> hi = bf16x2(a, b) and lo = bf16x2(a - hi.a, b - hi.b).
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float ra = a - __low2float(h), rb = b - __high2float(h);
    memcpy(&hi, &h, 4);
    lo = pack_bf16(ra, rb);
}

// Block-wide int64 sum over kThreads threads (all threads must call).
__device__ __forceinline__ long long block_sum_ll(long long v, long long* scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[warp] = v;
    __syncthreads();
    long long s = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += scratch[w];
    return s;
}

// Logical token position of sequence `seq` -> physical pool row, or -1.
__device__ __forceinline__ long long map_position(const smla_decode_args& a, long long pos, int seq) {
    if (pos < 0) return -1;
    long long phys;
    if (a.block_table == nullptr) {
        phys = pos;
    } else {
        const long long page = pos >> 6;
        if (page >= a.pages_per_seq) return -1;
        const int pid = __ldg(a.block_table + (size_t)seq * (size_t)a.pages_per_seq + (size_t)page);
        if (pid < 0) return -1;
        phys = (long long)pid * SMLA_PAGE_SIZE + (pos & (SMLA_PAGE_SIZE - 1));  // 64-bit
    }
    return phys < a.n_main ? phys : -1;
}

// Number of 64-entry tiles of row r: top-k slots, window, compressed groups.
__device__ __forceinline__ int row_tiles(const smla_decode_args& a, int r, uint32_t& err) {
    int t = ceil_div_i(a.topk, kBK);
    if (a.swa_len != nullptr) {
        int w = __ldg(a.swa_len + r);
        if (w < 0) { err |= SMLA_DEV_BAD_LENGTH; w = 0; }
        t += ceil_div_i(w, kBK);
    }
    if (a.cmp_len != nullptr) {
        int c = __ldg(a.cmp_len + r);
        if (c < 0) { err |= SMLA_DEV_BAD_LENGTH; c = 0; }
        t += ceil_div_i(c, kBK);
    }
    return t;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
smla_decode_kernel(const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(smem);
    const smla_decode_args& a = p.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t peer = crank ^ 1u;
    const int unit = blockIdx.x >> 1;
    const int R = a.num_rows, H = a.num_heads;

    const uint32_t bar_mma = sb + kOffBar, bar_full = sb + kOffBar + 8, bar_empty = sb + kOffBar + 16;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc);
    long long* red = reinterpret_cast<long long*>(smem + kOffMisc + 64);
    int* s_tiles = reinterpret_cast<int*>(smem + kOffTiles);
    int* s_prefix = reinterpret_cast<int*>(smem + kOffPrefix);
    const uint8_t** slot_e = reinterpret_cast<const uint8_t**>(smem + kOffSlotE);
    const uint8_t** slot_s = reinterpret_cast<const uint8_t**>(smem + kOffSlotS);

    uint32_t err = 0;

    if (tid == 0) {
        mbar_init(bar_mma, 1);
        mbar_init(bar_full, kThreads);
        mbar_init(bar_empty, kThreads);
        fence_mbar_init_cluster();
    }
    if (warp == 0) {
        tmem_alloc(sb + kOffMisc, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    // ---- in-kernel split plan (identical in every CTA; reads live lengths) ----
    // tiles_r per row; smallest chunk c with sum_r max(1, ceil(tiles_r / c)) <= units;
    // row r gets s_r = ceil(tiles_r / ceil(tiles_r / ceil(tiles_r / c))) splits.
    uint32_t plan_err = 0;
    int local_max = 0;
    for (int r = tid; r < R; r += kThreads) {
        const int t = row_tiles(a, r, plan_err);
        s_tiles[r] = t;
        local_max = max(local_max, t);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local_max = max(local_max, __shfl_xor_sync(0xffffffffu, local_max, o));
    __syncthreads();
    if (lane == 0) red[8 + warp] = local_max;
    __syncthreads();
    int max_t = 1;
    for (int w = 0; w < kThreads / 32; ++w) max_t = max(max_t, (int)red[8 + w]);
    int lo = 1, hi = max_t;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        long long cnt = 0;
        for (int r = tid; r < R; r += kThreads) cnt += max(1, ceil_div_i(s_tiles[r], mid));
        cnt = block_sum_ll(cnt, red);
        if (cnt <= p.units) hi = mid; else lo = mid + 1;
    }
    const int chunk = lo;
    // per-row split counts -> exclusive prefix (blocked scan: thread i owns rows [i*per, (i+1)*per))
    const int per = (R + kThreads - 1) / kThreads;
    int my_sum = 0;
    for (int r = tid * per; r < min(R, (tid + 1) * per); ++r) {
        const int t = s_tiles[r];
        int s = max(1, ceil_div_i(t, chunk));
        if (t > 0) s = ceil_div_i(t, ceil_div_i(t, s));
        my_sum += s;
    }
    int incl = my_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    __syncthreads();
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += (int)red[w];
    int run = base + incl - my_sum;
    for (int r = tid * per; r < min(R, (tid + 1) * per); ++r) {
        s_prefix[r] = run;
        const int t = s_tiles[r];
        int s = max(1, ceil_div_i(t, chunk));
        if (t > 0) s = ceil_div_i(t, ceil_div_i(t, s));
        run += s;
    }
    if (tid == kThreads - 1) s_prefix[R] = run;
    __syncthreads();
    const int total_units = s_prefix[R];

    // my unit -> (row, split)
    int row = -1, split = 0, s_r = 1, row_u0 = 0, t_begin = 0, t_end = 0;
    if (unit < total_units) {
        int l2 = 0, h2 = R - 1;  // last r with prefix[r] <= unit
        while (l2 < h2) {
            const int mid = (l2 + h2 + 1) >> 1;
            if (s_prefix[mid] <= unit) l2 = mid; else h2 = mid - 1;
        }
        row = l2;
        row_u0 = s_prefix[row];
        s_r = s_prefix[row + 1] - row_u0;
        split = unit - row_u0;
        const int T = s_tiles[row];
        const int tps = T > 0 ? ceil_div_i(T, s_r) : 0;
        t_begin = min(T, split * tps);
        t_end = min(T, t_begin + tps);
    }
    if (blockIdx.x == 0 && plan_err) err |= plan_err;

    bool aborted = false;
    if (row >= 0) {
        const int r = row;
        const int seq = a.row_seq != nullptr ? __ldg(a.row_seq + r) : r;
        const int nmt = ceil_div_i(a.topk, kBK);
        int swa_len = 0, swa_start = 0, cmp_len = 0;
        long long cmp_start = 0;
        if (a.swa_len != nullptr) { swa_len = max(0, __ldg(a.swa_len + r)); swa_start = __ldg(a.swa_start + r); }
        if (a.cmp_len != nullptr) { cmp_len = max(0, __ldg(a.cmp_len + r)); cmp_start = __ldg(a.cmp_start + r); }
        const int nst = ceil_div_i(swa_len, kBK);

        // ---- Q half -> shared memory (K-major, 128-byte swizzle) ----
        {
            const uint16_t* qn = static_cast<const uint16_t*>(a.q_nope) + (size_t)r * H * SMLA_NOPE_DIMS;
            const uint16_t* qr = static_cast<const uint16_t*>(a.q_rope) + (size_t)r * H * SMLA_ROPE_DIMS;
            for (int i = tid; i < 128 * 32; i += kThreads) {
                const int h = i >> 5, k = i & 31;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (h < H) {
                    if (crank == 0) v = __ldg(reinterpret_cast<const uint4*>(qn + (size_t)h * SMLA_NOPE_DIMS + k * 8));
                    else if (k < 24) v = __ldg(reinterpret_cast<const uint4*>(qn + (size_t)h * SMLA_NOPE_DIMS + 256 + k * 8));
                    else v = __ldg(reinterpret_cast<const uint4*>(qr + (size_t)h * SMLA_ROPE_DIMS + (k - 24) * 8));
                }
                st_shared_v4(sb + kOffQ + (k >> 3) * 16384 + sw128_offset(h, k & 7), v.x, v.y, v.z, v.w);
            }
        }

        const float qscale = a.sm_scale * kLog2e;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t idesc_qk = idesc_bf16_f32(128, kBK, false, false);
        const uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
        const uint32_t peer_sin = map_to_rank(sb + kOffSin, peer);
        const uint32_t peer_full = map_to_rank(bar_full, peer);
        const uint32_t peer_empty = map_to_rank(bar_empty, peer);
        uint32_t ph_mma = 0, ph_full = 0, ph_empty = 0;
        float m2 = -INFINITY, lsum = 0.f;
        bool o_init = false;
        bool bad = false;

        for (int t = t_begin; t < t_end; ++t) {
            // ---- resolve the 64 slots of this tile ----
            if (tid < kBK) {
                const uint8_t* ep = nullptr;
                const uint8_t* sp = nullptr;
                if (t < nmt) {
                    const int j = t * kBK + tid;
                    if (j < a.topk) {
                        const int idx = __ldg(a.main_idx + (size_t)r * a.topk + j);
                        if (idx != -1) {
                            const long long phys = map_position(a, idx, seq);
                            if (phys >= 0) {
                                ep = static_cast<const uint8_t*>(a.kv_pool) + phys * SMLA_ENTRY_BYTES;
                                sp = static_cast<const uint8_t*>(a.kv_scales) + phys * SMLA_SCALE_BYTES;
                            } else if (crank == 0) {
                                err |= SMLA_DEV_BAD_INDEX;
                            }
                        }
                    }
                } else if (t < nmt + nst) {
                    const int j = (t - nmt) * kBK + tid;
                    if (j < swa_len) {
                        const long long phys = map_position(a, (long long)swa_start + j, seq);
                        if (phys >= 0) {
                            ep = static_cast<const uint8_t*>(a.kv_pool) + phys * SMLA_ENTRY_BYTES;
                            sp = static_cast<const uint8_t*>(a.kv_scales) + phys * SMLA_SCALE_BYTES;
                        } else if (crank == 0) {
                            err |= SMLA_DEV_BAD_INDEX;
                        }
                    }
                } else {
                    const int j = (t - nmt - nst) * kBK + tid;
                    if (j < cmp_len) {
                        const long long phys = cmp_start + j;
                        if (phys >= 0 && phys < a.n_cmp) {
                            ep = static_cast<const uint8_t*>(a.cmp_pool) + phys * SMLA_ENTRY_BYTES;
                            sp = static_cast<const uint8_t*>(a.cmp_scales) + phys * SMLA_SCALE_BYTES;
                        } else if (crank == 0) {
                            err |= SMLA_DEV_BAD_CMP;
                        }
                    }
                }
                slot_e[tid] = ep;
                slot_s[tid] = sp;
                const uint32_t vb = __ballot_sync(0xffffffffu, ep != nullptr);
                if (lane == 0) misc[4 + warp] = vb;
            }
            __syncthreads();

            // ---- gather + dequantise this CTA's half of each entry ----
            {
                const int nch = crank == 0 ? 16 : 20;
                for (int i = tid; i < kBK * nch; i += kThreads) {
                    const int e = i / nch, k = i - e * nch;
                    const uint8_t* ep = slot_e[e];
                    if (crank == 0 || k < 12) {
                        const int atom = k >> 2, kk = (k & 3) * 2;
                        uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                        if (ep != nullptr) {
                            const int byte0 = (crank == 0 ? 0 : 256) + 16 * k;
                            const uint4 raw = ld_global_nc_v4(ep + byte0);
                            const float sc = ue8m0_to_f32(__ldg(slot_s[e] + (byte0 >> 6)));
                            dequant16(raw, sc, o);
                        }
                        const uint32_t dst = sb + kOffX + atom * 8192;
                        st_shared_v4(dst + sw128_offset(e, kk), o[0], o[1], o[2], o[3]);
                        st_shared_v4(dst + sw128_offset(e, kk + 1), o[4], o[5], o[6], o[7]);
                    } else {
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (ep != nullptr) v = ld_global_nc_v4(ep + SMLA_NOPE_DIMS + 16 * (k - 12));
                        st_shared_v4(sb + kOffX + 3 * 8192 + sw128_offset(e, k - 12), v.x, v.y, v.z, v.w);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(bad)) { aborted = true; break; }

            // ---- partial QK over this CTA's 256 dims ----
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t ad = sdesc_sw128(sb + kOffQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sb + kOffX + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + kTmemS, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar_mma);
            }
            __syncwarp();
            if (!mbar_wait_bounded<false>(bar_mma, ph_mma, kWaitNs)) bad = true;
            ph_mma ^= 1u;
            tc_fence_after();

            float s[64];
            {
                uint32_t v0[32], v1[32];
                tmem_ld32(tmem + kTmemS + lane_base, v0);
                tmem_ld32(tmem + kTmemS + lane_base + 32, v1);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) { s[j] = __uint_as_float(v0[j]); s[32 + j] = __uint_as_float(v1[j]); }
            }

            // ---- exchange partial scores with the peer CTA ----
            if (t > t_begin) {
                if (!mbar_wait_bounded<true>(bar_empty, ph_empty, kWaitNs)) bad = true;
                ph_empty ^= 1u;
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint32_t addr = peer_sin + tid * 256 + ((q ^ (tid & 15)) << 4);
                st_cluster_v4(addr, s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
            }
            mbar_arrive_remote(peer_full);
            if (!mbar_wait_bounded<true>(bar_full, ph_full, kWaitNs)) bad = true;
            ph_full ^= 1u;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint4 v = ld_shared_v4(sb + kOffSin + tid * 256 + ((q ^ (tid & 15)) << 4));
                s[4 * q] += __uint_as_float(v.x);
                s[4 * q + 1] += __uint_as_float(v.y);
                s[4 * q + 2] += __uint_as_float(v.z);
                s[4 * q + 3] += __uint_as_float(v.w);
            }
            mbar_arrive_remote(peer_empty);

            // ---- online softmax (log2 domain), P -> shared memory ----
            const uint32_t vm0 = misc[4], vm1 = misc[5];
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const bool valid = ((j < 32 ? vm0 >> j : vm1 >> (j - 32)) & 1u) != 0u;
                s[j] = valid ? s[j] * qscale : -INFINITY;
                mt = fmaxf(mt, s[j]);
            }
            const float m_new = fmaxf(m2, mt);
            const float alpha = (m2 == -INFINITY) ? 0.f : exp2f(m2 - m_new);
            float ps = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                s[j] = (s[j] == -INFINITY) ? 0.f : exp2f(s[j] - m_new);
                ps += s[j];
            }
            lsum = lsum * alpha + ps;
            m2 = m_new;
            // P = hi + lo, both bf16: the pair carries p to ~2^-17 relative, so
            // the PV product keeps fp32-level accuracy even when large V values
            // of nearly tied entries cancel.
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) split_bf16x2(s[8 * q + 2 * k], s[8 * q + 2 * k + 1], hi[k], lo[k]);
                st_shared_v4(sb + kOffP + sw128_offset(tid, q), hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(sb + kOffPlo + sw128_offset(tid, q), lo[0], lo[1], lo[2], lo[3]);
            }
            // rescale the running O when the max moved
            if (o_init && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem + kTmemO + lane_base + 32 * c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
                    tmem_st32(tmem + kTmemO + lane_base + 32 * c, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(bad)) { aborted = true; break; }

            // ---- PV into this CTA's half of O ----
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_sw128(sb + kOffP + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sb + kOffX + kk * 2048, kBK * 128, 1024);
                    mma_bf16_ss(tmem + kTmemO, ad, bd, idesc_pv, (o_init || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_sw128(sb + kOffPlo + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sb + kOffX + kk * 2048, kBK * 128, 1024);
                    mma_bf16_ss(tmem + kTmemO, ad, bd, idesc_pv, 1u);
                }
                mma_commit(bar_mma);
            }
            __syncwarp();
            if (!mbar_wait_bounded<false>(bar_mma, ph_mma, kWaitNs)) bad = true;
            ph_mma ^= 1u;
            tc_fence_after();
            o_init = true;
        }
        if (!aborted && __syncthreads_or(bad)) aborted = true;

        // ---- finish: final bf16 output, or fp32 partial + last-arriver merge ----
        const int h = tid;
        const float sink2 = (a.sink != nullptr && h < H) ? __ldg(a.sink + h) * kLog2e : -INFINITY;
        if (aborted) {
            err |= SMLA_DEV_TIMEOUT;
        } else if (s_r == 1) {
            const float M = fmaxf(m2, sink2);
            float oscale = 0.f, lse = -INFINITY;
            if (M != -INFINITY) {
                const float wm = (m2 == -INFINITY) ? 0.f : exp2f(m2 - M);
                const float wsink = (sink2 == -INFINITY) ? 0.f : exp2f(sink2 - M);
                const float Z = lsum * wm + wsink;
                oscale = Z > 0.f ? wm / Z : 0.f;
                lse = (M + log2f(Z)) * kLn2;
            }
            if (lsum == 0.f) lse = (a.sink != nullptr && h < H) ? __ldg(a.sink + h) : -INFINITY;  // sink only, exactly
            uint16_t* outp = static_cast<uint16_t*>(a.out) + ((size_t)r * H + (h < H ? h : 0)) * SMLA_HEAD_DIM + 256 * crank;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                if (o_init) {
                    tmem_ld32(tmem + kTmemO + lane_base + 32 * c, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0u;
                }
                if (h < H) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(v[8 * q]) * oscale, __uint_as_float(v[8 * q + 1]) * oscale);
                        w.y = pack_bf16(__uint_as_float(v[8 * q + 2]) * oscale, __uint_as_float(v[8 * q + 3]) * oscale);
                        w.z = pack_bf16(__uint_as_float(v[8 * q + 4]) * oscale, __uint_as_float(v[8 * q + 5]) * oscale);
                        w.w = pack_bf16(__uint_as_float(v[8 * q + 6]) * oscale, __uint_as_float(v[8 * q + 7]) * oscale);
                        *reinterpret_cast<uint4*>(outp + 32 * c + 8 * q) = w;
                    }
                }
            }
            if (crank == 0 && a.lse != nullptr && h < H) a.lse[(size_t)r * H + h] = lse;
        } else {
            // partial: unnormalised O (this half), and (m, l) per half
            const size_t ub = (size_t)unit;
            float* po = p.po + (ub * H + (h < H ? h : 0)) * SMLA_HEAD_DIM + 256 * crank;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + kTmemO + lane_base + 32 * c, v);
                tmem_wait_ld();
                if (h < H) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcg(reinterpret_cast<float4*>(po + 32 * c + 4 * q),
                               make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
                }
            }
            if (h < H) __stcg(p.ml + (ub * 2 + crank) * H + h, make_float2(m2, lsum));
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const uint32_t old = atomicAdd(p.counters + 2 * r + crank, 1u);
                misc[2] = (old == (uint32_t)(s_r - 1)) ? 1u : 0u;
            }
            __syncthreads();
            if (misc[2] != 0u) {
                __threadfence();
                // merge the s_r partials of (row r, this half) in split order
                if (h < H) {
                    float M = sink2;
                    for (int i = 0; i < s_r; ++i) M = fmaxf(M, __ldcg(p.ml + ((size_t)(row_u0 + i) * 2 + crank) * H + h).x);
                    float Z = 0.f, lall = 0.f;
                    if (M != -INFINITY) {
                        Z = (sink2 == -INFINITY) ? 0.f : exp2f(sink2 - M);
                        for (int i = 0; i < s_r; ++i) {
                            const float2 ml = __ldcg(p.ml + ((size_t)(row_u0 + i) * 2 + crank) * H + h);
                            if (ml.x != -INFINITY) Z += ml.y * exp2f(ml.x - M);
                            lall += ml.y;
                        }
                    }
                    const float inv = Z > 0.f ? 1.f / Z : 0.f;
                    uint16_t* outp = static_cast<uint16_t*>(a.out) + ((size_t)r * H + h) * SMLA_HEAD_DIM + 256 * crank;
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        float acc[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
                        for (int i = 0; i < s_r; ++i) {
                            const size_t u = (size_t)(row_u0 + i);
                            const float mi = __ldcg(p.ml + (u * 2 + crank) * H + h).x;
                            if (mi == -INFINITY) continue;
                            const float w = exp2f(mi - M) * inv;
                            const float* src = p.po + (u * H + h) * SMLA_HEAD_DIM + 256 * crank + 32 * c;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 v = __ldcg(reinterpret_cast<const float4*>(src + 4 * q));
                                acc[4 * q] += w * v.x;
                                acc[4 * q + 1] += w * v.y;
                                acc[4 * q + 2] += w * v.z;
                                acc[4 * q + 3] += w * v.w;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 wv;
                            wv.x = pack_bf16(acc[8 * q], acc[8 * q + 1]);
                            wv.y = pack_bf16(acc[8 * q + 2], acc[8 * q + 3]);
                            wv.z = pack_bf16(acc[8 * q + 4], acc[8 * q + 5]);
                            wv.w = pack_bf16(acc[8 * q + 6], acc[8 * q + 7]);
                            *reinterpret_cast<uint4*>(outp + 32 * c + 8 * q) = wv;
                        }
                    }
                    if (crank == 0 && a.lse != nullptr) {
                        float lse = (M == -INFINITY || Z <= 0.f) ? -INFINITY : (M + log2f(Z)) * kLn2;
                        if (lall == 0.f) lse = a.sink != nullptr ? __ldg(a.sink + h) : -INFINITY;  // sink only, exactly
                        a.lse[(size_t)r * H + h] = lse;
                    }
                }
                if (tid == 0) atomicExch(p.counters + 2 * r + crank, 0u);
            }
        }
    }

    if (err != 0u) atomicOr(p.err, err);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    cluster_sync();
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
namespace {
std::atomic<int> g_attr_done[64];
std::mutex g_attr_mu;

cudaError_t ensure_kernel_attrs(int dev) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_attr_done[dev].load(std::memory_order_acquire) == 1) return cudaSuccess;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (g_attr_done[dev].load(std::memory_order_relaxed) == 1) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(smla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_done[dev].store(1, std::memory_order_release);
    return cudaSuccess;
}
}  // namespace

smla_status launch_decode(const smla_decode_args* args, void* workspace, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
    if (ensure_kernel_attrs(dev) != cudaSuccess) return SMLA_ERR_CUDA;
    const WorkspaceLayout L = workspace_layout(args->num_rows, args->num_heads, args->num_splits);
    KParams kp;
    kp.a = *args;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    kp.err = reinterpret_cast<uint32_t*>(ws + L.off_err);
    kp.counters = reinterpret_cast<uint32_t*>(ws + L.off_counters);
    kp.ml = reinterpret_cast<float2*>(ws + L.off_ml);
    kp.po = reinterpret_cast<float*>(ws + L.off_po);
    kp.units = args->num_rows * args->num_splits;
    const dim3 grid((unsigned)(2 * kp.units)), block(kThreads);
    smla_decode_kernel<<<grid, block, kSmemBytes, stream>>>(kp);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
