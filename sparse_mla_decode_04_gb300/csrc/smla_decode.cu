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
// GB300 design.  A work unit is (row, split) and runs on a CTA pair (cluster
// of 2); CTA c owns dims [256c, 256c+256) of the 512-wide head dim, because O
// for 128 heads x 512 dims in fp32 would fill a whole SM's TMEM.  The grid is
// persistent: each cluster walks its share of the units.  Inside a CTA the
// work is split over warp roles that hand 64-entry tiles along mbarrier rings:
//
//   producer warps (4)   resolve a tile's slots (top-k index -> page table ->
//                        64-bit row; window; compressed) and issue one bulk
//                        copy per valid entry of this CTA's half of its bytes
//                        into a 4-stage raw ring, plus the entry's scale codes;
//   dequant warps (4)    raw ring -> bf16 tile (e4m3 x 2^(code-127), exact) in
//                        a 3-stage ring of 128-byte-swizzled tiles, each of
//                        which is the K-major B operand of QK and the MN-major
//                        B operand of PV;
//   MMA warp (1 thread)  QK(t) = Q . X(t)^T on tcgen05 (M = 128 heads, N = 64,
//                        K = 256, A = Q from TMEM), then PV(t-1);
//   softmax warps (4)    one thread per head (TMEM lane): partial scores are
//                        swapped with the peer CTA through distributed shared
//                        memory and summed (fp32 addition commutes, so both CTAs
//                        hold identical scores), online softmax with a
//                        conditional rescale, and P written back into the score
//                        columns of TMEM as a bf16 pair hi = bf16(p),
//                        lo = bf16(p - hi) for PV (A from TMEM).  A single bf16
//                        P (8-bit mantissa) is not enough: with V near 600 in
//                        magnitude, nearly tied entries whose V values cancel
//                        would carry errors near 1.  The lo half is skipped on
//                        tiles where a running bound (sum |lo| x max |V|) shows
//                        its total effect on every head's output stays within
//                        2^-9; on peaked softmaxes most tiles qualify.
//
// TMEM (512 columns): O [0, 256), two score/P buffers [256, 384), Q [384, 512).
// Heads beyond num_heads are zero-padded up to the MMA's M = 128.
#include <algorithm>
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

constexpr int kBK = 64;               // entries per tile
constexpr int kNR = 4;                // raw-byte ring stages
constexpr int kNX = 3;                // bf16 tile ring stages
constexpr int kSoftmaxWarps = 4;      // warps 0-3: one thread per head
constexpr int kProducerWarp0 = 4;     // warps 4-7: one producer per raw stage
constexpr int kNumProducers = kNR;
constexpr int kMmaWarp = 8;
constexpr int kDequantWarp0 = 9;      // warps 9-12
constexpr int kNumDequantWarps = 4;
constexpr int kWarps = 13;
constexpr int kThreads = 32 * kWarps;
constexpr int kHeadsPad = 128;
constexpr int kMaxUnitsPerCluster = 32;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;        // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;      // score / P buffers: [256, 320), [320, 384)
constexpr uint32_t kTmemQ = 384;      // Q half, bf16 packed: [384, 512)
constexpr uint64_t kWaitNs = 2000000000ull;  // bounded-wait limit (2 s)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow to 2^8 before O is rescaled
// The lo half of P is skipped on a tile only while, for every head, the bound
// on everything skipped so far stays within kLoBudget of the running softmax
// denominator: the output error from skipping is then at most kLoBudget.
constexpr float kLoBudget = 1.0f / 512.0f;

constexpr uint32_t kRawEntryBytes = 320;   // CTA0 uses 256 of them, CTA1 all 320
constexpr uint32_t kXStageBytes = 4 * kBK * 128;           // 32 KB
constexpr uint32_t kRawStageBytes = kBK * kRawEntryBytes;  // 20 KB

// Shared-memory layout (offsets from a 1024-byte-aligned base).
constexpr uint32_t kOffX = 0;                                   // [kNX][4 atoms][64][128 B]
constexpr uint32_t kOffRaw = kOffX + kNX * kXStageBytes;        // [kNR][64][320 B]
constexpr uint32_t kOffRawSc = kOffRaw + kNR * kRawStageBytes;  // [kNR][64] u64 scale codes
constexpr uint32_t kOffSin = kOffRawSc + kNR * kBK * 8;         // peer's partial S [128][64] f32 (32 KB)
constexpr uint32_t kOffRawMask = kOffSin + 32768;               // [kNR] u64 valid masks
constexpr uint32_t kOffXMask = kOffRawMask + kNR * 8;           // [kNX] u64 valid masks
constexpr uint32_t kOffXVmax = kOffXMask + 32;                  // [kNX][4 dequant warps] f32 max |V| bound
constexpr uint32_t kOffVote = kOffXVmax + kNX * 16;             // [2][4 softmax warps] u32 lo-skip votes
constexpr uint32_t kOffBar = kOffVote + 32;                     // mbarriers
constexpr uint32_t kNumBars = 32;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;           // tmem base, flags, reductions
constexpr uint32_t kMiscBytes = 512;
constexpr uint32_t kOffUnits = kOffMisc + kMiscBytes;           // unit descriptors
constexpr uint32_t kSmemUsed = kOffUnits + kMaxUnitsPerCluster * 32;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;               // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
// The plan's per-row scratch (tiles[R], prefix[R+1]) aliases the exchange buffer
// during the prologue; a cluster barrier separates it from the first exchange.
static_assert(4 * (2 * SMLA_MAX_ROWS + 8) <= 32768, "plan scratch fits in the exchange buffer");

// mbarrier indices
enum : uint32_t {
    BAR_RAW_FULL = 0,                      // [kNR] producer -> dequant (1 arrival + tx bytes)
    BAR_RAW_EMPTY = BAR_RAW_FULL + kNR,    // [kNR] dequant -> producer (kNumDequantWarps)
    BAR_X_FULL = BAR_RAW_EMPTY + kNR,      // [kNX] dequant -> MMA, softmax (kNumDequantWarps)
    BAR_X_EMPTY = BAR_X_FULL + kNX,        // [kNX] MMA commit after PV
    BAR_S_FULL = BAR_X_EMPTY + kNX,        // [2] MMA commit after QK
    BAR_P_FULL = BAR_S_FULL + 2,           // [2] softmax -> MMA (kSoftmaxWarps)
    BAR_O_DONE = BAR_P_FULL + 2,           // MMA commit after each PV
    BAR_Q_READY = BAR_O_DONE + 1,          // softmax -> MMA, once per unit (kSoftmaxWarps)
    BAR_EX_FULL = BAR_Q_READY + 1,         // peer's partial S landed (kHeadsPad remote arrivals)
    BAR_EX_EMPTY = BAR_EX_FULL + 1,        // peer consumed our partial S (kHeadsPad remote arrivals)
    BAR_MMA_FINAL = BAR_EX_EMPTY + 1,      // teardown: all MMAs retired
    BAR_COUNT = BAR_MMA_FINAL + 1
};
static_assert(BAR_COUNT <= kNumBars, "barrier slots");

struct KParams {
    smla_decode_args a;
    uint32_t* err;
    uint32_t* counters;  // [SMLA_MAX_ROWS][2]
    float2* ml;          // [units][2][H]   (m in log2 units, l)
    float* po;           // [units][H][512] unnormalised fp32 O
    int units;           // num_rows * num_splits (work units of the plan)
};

struct UnitDesc {
    int row, s_r, row_u0, unit, t_begin, t_end, pad0, pad1;
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

// (a, b) -> hi = bf16x2(a, b) and lo = bf16x2(a - hi.a, b - hi.b).
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float ra = a - __low2float(h), rb = b - __high2float(h);
    memcpy(&hi, &h, 4);
    lo = pack_bf16(ra, rb);
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
            o[2 * i + j] = pack_bf16(__half2float(lo) * scale, __half2float(hi) * scale);
        }
    }
}

// Upper bound of |x| over 16 e4m3 codes: the 7-bit magnitude pattern of an
// e4m3 code orders like its value, so the largest pattern decodes to the
// largest magnitude.  The NaN pattern (0x7F) gives +inf (never skip).
__device__ __forceinline__ float e4m3x16_absmax(const uint4 v) {
    const uint32_t k = 0x7F7F7F7Fu;
    const uint32_t m4 = __vmaxu4(__vmaxu4(v.x & k, v.y & k), __vmaxu4(v.z & k, v.w & k));
    const uint32_t mb = max(max(m4 & 0xFFu, (m4 >> 8) & 0xFFu), max((m4 >> 16) & 0xFFu, m4 >> 24));
    if (mb == 0x7Fu) return INFINITY;
    const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)mb, __NV_E4M3);
    __half hv;
    memcpy(&hv, &hr, 2);
    return __half2float(hv);
}

// Upper bound of |x| over 8 bf16 values (NaN gives +inf).
__device__ __forceinline__ float bf16x8_absmax(const uint4 v) {
    const uint32_t k = 0x7FFF7FFFu;
    const uint32_t m2 = __vmaxu2(__vmaxu2(v.x & k, v.y & k), __vmaxu2(v.z & k, v.w & k));
    const uint32_t mh = max(m2 & 0xFFFFu, m2 >> 16);
    return mh > 0x7F80u ? INFINITY : __uint_as_float(mh << 16);
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

// Per-CTA state shared by the roles.
struct Ctx {
    uint32_t sb;              // shared base (1024-aligned)
    uint32_t tmem;            // TMEM base address
    uint32_t crank, peer;
    volatile uint32_t* abort; // set by any role whose bounded wait gave up
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, uint32_t i) { return c.sb + kOffBar + 8 * i; }

// Bounded wait that also gives up as soon as another role of this CTA aborted.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar(const Ctx& c, uint32_t bar, uint32_t parity) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if (global_timer_ns() - t0 > kWaitNs) {
            *c.abort = 1u;
            return false;
        }
    }
}

// The same wait, taken by a whole warp: the outcome is made warp-uniform so
// that the warp never splits around warp-synchronous code after a timeout.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar_warp(const Ctx& c, uint32_t bar, uint32_t parity) {
    const bool ok = wait_bar<kCluster>(c, bar, parity);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void st_shared_u64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared.b64 [%0], %1;" :: "r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_shared_u64(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Named barrier over the softmax warps only (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void softmax_bar() {
    asm volatile("bar.sync 1, %0;" :: "r"(kSoftmaxWarps * 32) : "memory");
}

// AND of `v` over the softmax warps (named barrier 1): every softmax thread
// reaches it exactly once per unit, whatever happened in the tile loop.
__device__ __forceinline__ bool softmax_all(bool v) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, 1, %2, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v), "r"(kSoftmaxWarps * 32) : "memory");
    return r != 0u;
}

// ---------------------------------------------------------------------------
// role: producer (one warp per raw stage; warp pw handles tiles g % kNR == pw)
// ---------------------------------------------------------------------------
__device__ void producer_role(const KParams& p, const Ctx& c, const UnitDesc* units, int n_units, int pw,
                              uint32_t& err) {
    const smla_decode_args& a = p.a;
    const int lane = threadIdx.x & 31;
    const uint32_t off = c.crank == 0 ? 0u : 256u;
    const uint32_t bytes = c.crank == 0 ? 256u : 320u;
    uint32_t g = 0;
    for (int ui = 0; ui < n_units; ++ui) {
        const UnitDesc d = units[ui];
        const int r = d.row;
        const int seq = a.row_seq != nullptr ? __ldg(a.row_seq + r) : r;
        const int nmt = ceil_div_i(a.topk, kBK);
        int swa_len = 0, swa_start = 0, cmp_len = 0;
        long long cmp_start = 0;
        if (a.swa_len != nullptr) { swa_len = max(0, __ldg(a.swa_len + r)); swa_start = __ldg(a.swa_start + r); }
        if (a.cmp_len != nullptr) { cmp_len = max(0, __ldg(a.cmp_len + r)); cmp_start = __ldg(a.cmp_start + r); }
        const int nst = ceil_div_i(swa_len, kBK);
        for (int t = d.t_begin; t < d.t_end; ++t, ++g) {
            if ((int)(g % kNR) != pw) continue;
            const uint32_t rs = g % kNR, rph = (g / kNR) & 1u;
            // resolve this lane's two slots
            const uint8_t* ep[2] = {nullptr, nullptr};
            const uint8_t* sp[2] = {nullptr, nullptr};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int slot = lane + 32 * k;
                long long phys = -1;
                bool cmp = false;
                if (t < nmt) {
                    const int j = t * kBK + slot;
                    if (j < a.topk) {
                        const int idx = __ldg(a.main_idx + (size_t)r * a.topk + j);
                        if (idx != -1) {
                            phys = map_position(a, idx, seq);
                            if (phys < 0) err |= SMLA_DEV_BAD_INDEX;
                        }
                    }
                } else if (t < nmt + nst) {
                    const int j = (t - nmt) * kBK + slot;
                    if (j < swa_len) {
                        phys = map_position(a, (long long)swa_start + j, seq);
                        if (phys < 0) err |= SMLA_DEV_BAD_INDEX;
                    }
                } else {
                    const int j = (t - nmt - nst) * kBK + slot;
                    if (j < cmp_len) {
                        cmp = true;
                        phys = cmp_start + j;
                        if (phys < 0 || phys >= a.n_cmp) {
                            err |= SMLA_DEV_BAD_CMP;
                            phys = -1;
                        }
                    }
                }
                if (phys >= 0) {
                    ep[k] = static_cast<const uint8_t*>(cmp ? a.cmp_pool : a.kv_pool) + phys * SMLA_ENTRY_BYTES;
                    sp[k] = static_cast<const uint8_t*>(cmp ? a.cmp_scales : a.kv_scales) + phys * SMLA_SCALE_BYTES;
                }
            }
            const uint32_t m0 = __ballot_sync(0xffffffffu, ep[0] != nullptr);
            const uint32_t m1 = __ballot_sync(0xffffffffu, ep[1] != nullptr);
            if (!wait_bar_warp<false>(c, bar_addr(c, BAR_RAW_EMPTY + rs), rph ^ 1u)) return;
            const uint32_t full = bar_addr(c, BAR_RAW_FULL + rs);
            if (lane == 0) mbar_expect_tx_only(full, (uint32_t)(__popc(m0) + __popc(m1)) * bytes);
            __syncwarp();
            const uint32_t raw = c.sb + kOffRaw + rs * kRawStageBytes;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (ep[k] != nullptr) bulk_g2s(raw + (lane + 32 * k) * kRawEntryBytes, ep[k] + off, bytes, full);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint2 sc = make_uint2(0u, 0u);
                if (sp[k] != nullptr) sc = ld_global_nc_v2(sp[k]);
                st_shared_u64(c.sb + kOffRawSc + (rs * kBK + lane + 32 * k) * 8,
                              (uint64_t)sc.x | ((uint64_t)sc.y << 32));
            }
            if (lane == 0) st_shared_u64(c.sb + kOffRawMask + rs * 8, (uint64_t)m0 | ((uint64_t)m1 << 32));
            __syncwarp();
            if (lane == 0) mbar_arrive_local(full);
        }
    }
}

// ---------------------------------------------------------------------------
// role: dequant (4 warps): raw ring -> bf16 swizzled tile ring
// ---------------------------------------------------------------------------
__device__ void dequant_role(const Ctx& c, const UnitDesc* units, int n_units, int dw) {
    const int lane = threadIdx.x & 31;
    const int dtid = dw * 32 + lane;
    const int nch = c.crank == 0 ? 16 : 20;
    uint32_t g = 0;
    for (int ui = 0; ui < n_units; ++ui) {
        const int n = units[ui].t_end - units[ui].t_begin;
        for (int i = 0; i < n; ++i, ++g) {
            const uint32_t rs = g % kNR, rph = (g / kNR) & 1u;
            const uint32_t xs = g % kNX, xph = (g / kNX) & 1u;
            if (!wait_bar_warp<false>(c, bar_addr(c, BAR_RAW_FULL + rs), rph)) return;
            if (!wait_bar_warp<false>(c, bar_addr(c, BAR_X_EMPTY + xs), xph ^ 1u)) return;
            const uint64_t mask = ld_shared_u64(c.sb + kOffRawMask + rs * 8);
            const uint32_t raw = c.sb + kOffRaw + rs * kRawStageBytes;
            const uint32_t xb = c.sb + kOffX + xs * kXStageBytes;
            float vbound = 0.f;  // >= |x| for every value this thread wrote
            for (int idx = dtid; idx < kBK * nch; idx += kNumDequantWarps * 32) {
                const int e = idx / nch, k = idx - e * nch;
                const bool valid = ((mask >> e) & 1ull) != 0ull;
                if (c.crank == 0 || k < 12) {
                    const int atom = k >> 2, kk = (k & 3) * 2;
                    uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    if (valid) {
                        const uint4 v = ld_shared_v4(raw + e * kRawEntryBytes + 16 * k);
                        const uint32_t byte0 = (c.crank == 0 ? 0u : 256u) + 16u * (uint32_t)k;
                        const uint32_t code = ld_shared_u8(c.sb + kOffRawSc + (rs * kBK + e) * 8 + (byte0 >> 6));
                        const float scale = ue8m0_to_f32(code);
                        dequant16(v, scale, o);
                        const float bnd = e4m3x16_absmax(v) * scale;
                        vbound = (bnd > vbound || bnd != bnd) ? (bnd != bnd ? INFINITY : bnd) : vbound;
                    }
                    const uint32_t dst = xb + atom * (kBK * 128);
                    st_shared_v4(dst + sw128_offset(e, kk), o[0], o[1], o[2], o[3]);
                    st_shared_v4(dst + sw128_offset(e, kk + 1), o[4], o[5], o[6], o[7]);
                } else {
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (valid) v = ld_shared_v4(raw + e * kRawEntryBytes + 16 * k);
                    vbound = fmaxf(vbound, bf16x8_absmax(v));
                    st_shared_v4(xb + 3 * (kBK * 128) + sw128_offset(e, k - 12), v.x, v.y, v.z, v.w);
                }
            }
            if (dtid == 0) st_shared_u64(c.sb + kOffXMask + xs * 8, mask);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) vbound = fmaxf(vbound, __shfl_xor_sync(0xffffffffu, vbound, o));
            if (lane == 0)
                asm volatile("st.shared.f32 [%0], %1;" :: "r"(c.sb + kOffXVmax + (xs * 4 + dw) * 4), "f"(vbound) : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_local(bar_addr(c, BAR_X_FULL + xs));
                mbar_arrive_local(bar_addr(c, BAR_RAW_EMPTY + rs));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// role: MMA issuer (one thread)
// ---------------------------------------------------------------------------
// PV(j): O += P(j) . X(j), with P as the hi then lo bf16 pair from TMEM.
__device__ __forceinline__ bool issue_pv(const Ctx& c, uint32_t j, bool first_of_unit) {
    const uint32_t sb = j & 1u, xs = j % kNX;
    if (!wait_bar<false>(c, bar_addr(c, BAR_P_FULL + sb), (j >> 1) & 1u)) return false;
    tc_fence_after();
    const uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
    const uint32_t xb = c.sb + kOffX + xs * kXStageBytes;
    const uint32_t tp = c.tmem + kTmemS + sb * 64;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bd = sdesc_sw128(xb + kk * 2048, kBK * 128, 1024);
        mma_bf16_ts(c.tmem + kTmemO, tp + kk * 8, bd, idesc_pv, (first_of_unit && kk == 0) ? 0u : 1u);
    }
    uint32_t votes = 1u;
#pragma unroll
    for (int w = 0; w < kSoftmaxWarps; ++w) {
        uint32_t v;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(c.sb + kOffVote + (sb * 4 + w) * 4) : "memory");
        votes &= v;
    }
    if (votes == 0u) {  // some head needs the lo half of P on this tile
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc_sw128(xb + kk * 2048, kBK * 128, 1024);
            mma_bf16_ts(c.tmem + kTmemO, tp + 32 + kk * 8, bd, idesc_pv, 1u);
        }
    }
    mma_commit(bar_addr(c, BAR_X_EMPTY + xs));
    mma_commit(bar_addr(c, BAR_O_DONE));
    return true;
}

__device__ void mma_role(const Ctx& c, const UnitDesc* units, int n_units) {
    const uint32_t idesc_qk = idesc_bf16_f32(128, kBK, false, false);
    uint32_t g = 0;
    bool ok = true;
    for (int ui = 0; ui < n_units && ok; ++ui) {
        const int n = units[ui].t_end - units[ui].t_begin;
        if (!wait_bar<false>(c, bar_addr(c, BAR_Q_READY), (uint32_t)ui & 1u)) break;
        tc_fence_after();
        const uint32_t g0 = g;
        for (int i = 0; i < n; ++i, ++g) {
            const uint32_t xs = g % kNX;
            if (!wait_bar<false>(c, bar_addr(c, BAR_X_FULL + xs), (g / kNX) & 1u)) { ok = false; break; }
            tc_fence_after();
            const uint32_t xb = c.sb + kOffX + xs * kXStageBytes;
            const uint32_t ts = c.tmem + kTmemS + (g & 1u) * 64;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t bd = sdesc_sw128(xb + (kk >> 2) * (kBK * 128) + (kk & 3) * 32, 16, 1024);
                mma_bf16_ts(ts, c.tmem + kTmemQ + kk * 8, bd, idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar_addr(c, BAR_S_FULL + (g & 1u)));
            if (i > 0 && !issue_pv(c, g - 1, (g - 1) == g0)) { ok = false; break; }
        }
        if (ok && n > 0 && !issue_pv(c, g - 1, (g - 1) == g0)) ok = false;
    }
    // retire every MMA before TMEM is released
    mma_commit(bar_addr(c, BAR_MMA_FINAL));
    mbar_wait_bounded<false>(bar_addr(c, BAR_MMA_FINAL), 0, kWaitNs);
}

// ---------------------------------------------------------------------------
// role: softmax / epilogue (warps 0-3, thread = head = TMEM lane)
// ---------------------------------------------------------------------------
__device__ void softmax_role(const KParams& p, const Ctx& c, const UnitDesc* units, int n_units, uint32_t& err) {
    const smla_decode_args& a = p.a;
    const int h = threadIdx.x;  // 0..127
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = a.num_heads;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float qscale = a.sm_scale * kLog2e;
    const float sink2 = (a.sink != nullptr && h < H) ? __ldg(a.sink + h) * kLog2e : -INFINITY;
    const uint32_t peer_sin = map_to_rank(c.sb + kOffSin, c.peer);
    const uint32_t peer_full = map_to_rank(bar_addr(c, BAR_EX_FULL), c.peer);
    const uint32_t peer_empty = map_to_rank(bar_addr(c, BAR_EX_EMPTY), c.peer);
    volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(
        static_cast<uint8_t*>(__cvta_shared_to_generic(c.sb + kOffMisc + 12)));  // misc[3]
    uint32_t g = 0, pv = 0, ex = 0;
    bool ok = true;

    for (int ui = 0; ui < n_units && ok; ++ui) {
        const UnitDesc d = units[ui];
        const int r = d.row;
        const int n = d.t_end - d.t_begin;
        // ---- Q half of this row -> TMEM columns [384, 512) (bf16 pairs) ----
        {
            const size_t hq = (size_t)r * H + (h < H ? h : 0);
            const uint16_t* qn = static_cast<const uint16_t*>(a.q_nope) + hq * SMLA_NOPE_DIMS;
            const uint16_t* qr = static_cast<const uint16_t*>(a.q_rope) + hq * SMLA_ROPE_DIMS;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {  // 4 x 32 columns = 256 dims
                uint32_t v[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int k = cc * 8 + q;  // 16-byte chunk of this CTA's 256 dims
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (h < H) {
                        if (c.crank == 0) w = __ldg(reinterpret_cast<const uint4*>(qn + k * 8));
                        else if (k < 24) w = __ldg(reinterpret_cast<const uint4*>(qn + 256 + k * 8));
                        else w = __ldg(reinterpret_cast<const uint4*>(qr + (k - 24) * 8));
                    }
                    v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
                }
                tmem_st32(c.tmem + kTmemQ + lane_base + 32 * cc, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_Q_READY));
        }

        float m_used = -INFINITY, lsum = 0.f;
        float skipped = 0.f;  // bound on the lo-half contributions skipped so far (units of lsum)
        bool o_init = false;
        for (int i = 0; i < n; ++i, ++g) {
            const uint32_t sbuf = g & 1u;
            if (!wait_bar_warp<false>(c, bar_addr(c, BAR_S_FULL + sbuf), (g >> 1) & 1u)) { ok = false; break; }
            tc_fence_after();
            float s[64];
            {
                uint32_t v0[32], v1[32];
                tmem_ld32(c.tmem + kTmemS + sbuf * 64 + lane_base, v0);
                tmem_ld32(c.tmem + kTmemS + sbuf * 64 + lane_base + 32, v1);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) { s[j] = __uint_as_float(v0[j]); s[32 + j] = __uint_as_float(v1[j]); }
            }
            // ---- swap partial scores with the peer CTA ----
            if (ex > 0 && !wait_bar_warp<true>(c, bar_addr(c, BAR_EX_EMPTY), (ex - 1) & 1u)) { ok = false; break; }
#pragma unroll
            for (int q = 0; q < 16; ++q)
                st_cluster_v4(peer_sin + h * 256 + ((q ^ (h & 15)) << 4), s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
            mbar_arrive_remote(peer_full);
            if (!wait_bar_warp<true>(c, bar_addr(c, BAR_EX_FULL), ex & 1u)) { ok = false; break; }
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint4 v = ld_shared_v4(c.sb + kOffSin + h * 256 + ((q ^ (h & 15)) << 4));
                s[4 * q] += __uint_as_float(v.x);
                s[4 * q + 1] += __uint_as_float(v.y);
                s[4 * q + 2] += __uint_as_float(v.z);
                s[4 * q + 3] += __uint_as_float(v.w);
            }
            mbar_arrive_remote(peer_empty);
            ++ex;
            // ---- online softmax (log2 domain) with a conditional rescale ----
            // The tile's valid mask was written before its X_FULL arrival; X_FULL of
            // this tile cannot have advanced further (its stage is refilled only after
            // PV of this tile, which needs this thread's P).
            if (!wait_bar_warp<false>(c, bar_addr(c, BAR_X_FULL + g % kNX), (g / kNX) & 1u)) { ok = false; break; }
            const uint64_t vmask = ld_shared_u64(c.sb + kOffXMask + (g % kNX) * 8);
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                s[j] = ((vmask >> j) & 1ull) ? s[j] * qscale : -INFINITY;
                mt = fmaxf(mt, s[j]);
            }
            float m_new = m_used;
            if (m_used == -INFINITY || mt > m_used + kRescaleThreshold) m_new = fmaxf(m_used, mt);
            const float alpha = (m_used == -INFINITY) ? 0.f : exp2f(m_used - m_new);
            float ps = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                s[j] = (s[j] == -INFINITY) ? 0.f : exp2f(s[j] - m_new);
                ps += s[j];
            }
            lsum = lsum * alpha + ps;
            skipped *= alpha;
            const bool rescale = o_init && (m_new != m_used);
            m_used = m_new;
            // PV(g-1) must be done before O is touched or P(g) is handed over
            if (i > 0) {
                if (!wait_bar_warp<false>(c, bar_addr(c, BAR_O_DONE), pv & 1u)) { ok = false; break; }
                ++pv;
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? alpha : 1.f;
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(c.tmem + kTmemO + lane_base + 32 * cc, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * f);
                    tmem_st32(c.tmem + kTmemO + lane_base + 32 * cc, v);
                }
            }
            // ---- P -> TMEM score columns: hi in [0, 32), lo in [32, 64) ----
            float lo_abs = 0.f;
            {
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    split_bf16x2(s[2 * j], s[2 * j + 1], hi[j], lo[j]);
                    const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&hi[j]);
                    lo_abs += fabsf(s[2 * j] - __low2float(hv)) + fabsf(s[2 * j + 1] - __high2float(hv));
                }
                tmem_st32(c.tmem + kTmemS + sbuf * 64 + lane_base, hi);
                tmem_st32(c.tmem + kTmemS + sbuf * 64 + lane_base + 32, lo);
            }
            // vote on skipping the lo half: sum|lo| (x1.01 for its own rounding) x max|V| of the tile
            {
                const uint32_t vb = c.sb + kOffXVmax + (g % kNX) * 16;
                float vmax;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(vmax) : "r"(vb) : "memory");
#pragma unroll
                for (int w = 1; w < kNumDequantWarps; ++w) {
                    float t;
                    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(t) : "r"(vb + 4 * w) : "memory");
                    vmax = fmaxf(vmax, t);
                }
                const float cand = skipped + lo_abs * 1.0079f * vmax;
                const bool mine = (h >= H) || (cand <= kLoBudget * lsum);
                const bool warp_ok = __all_sync(0xffffffffu, mine);
                if (warp_ok) skipped = cand;  // counted even if another warp vetoes: conservative
                if (lane == 0)
                    asm volatile("st.shared.u32 [%0], %1;" :: "r"(c.sb + kOffVote + (sbuf * 4 + warp) * 4),
                                 "r"(warp_ok ? 1u : 0u) : "memory");
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_P_FULL + sbuf));
            o_init = true;
        }
        if (ok && n > 0) {
            if (!wait_bar_warp<false>(c, bar_addr(c, BAR_O_DONE), pv & 1u)) ok = false;
            ++pv;
            tc_fence_after();
        }
        if (!softmax_all(ok)) {  // uniform over the softmax warps from here on
            ok = false;
            *c.abort = 1u;
            break;
        }
        // ---- finish: final bf16 output, or fp32 partial + last-arriver merge ----
        if (d.s_r == 1) {
            const float M = fmaxf(m_used, sink2);
            float oscale = 0.f, lse = -INFINITY;
            if (M != -INFINITY) {
                const float wm = (m_used == -INFINITY) ? 0.f : exp2f(m_used - M);
                const float wsink = (sink2 == -INFINITY) ? 0.f : exp2f(sink2 - M);
                const float Z = lsum * wm + wsink;
                oscale = Z > 0.f ? wm / Z : 0.f;
                lse = (M + log2f(Z)) * kLn2;
            }
            if (lsum == 0.f) lse = (a.sink != nullptr && h < H) ? __ldg(a.sink + h) : -INFINITY;  // sink only, exactly
            uint16_t* outp = static_cast<uint16_t*>(a.out) + ((size_t)r * H + (h < H ? h : 0)) * SMLA_HEAD_DIM + 256 * c.crank;
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t v[32];
                if (o_init) {
                    tmem_ld32(c.tmem + kTmemO + lane_base + 32 * cc, v);
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
                        *reinterpret_cast<uint4*>(outp + 32 * cc + 8 * q) = w;
                    }
                }
            }
            if (c.crank == 0 && a.lse != nullptr && h < H) a.lse[(size_t)r * H + h] = lse;
        } else {
            const size_t ub = (size_t)d.unit;
            float* po = p.po + (ub * H + (h < H ? h : 0)) * SMLA_HEAD_DIM + 256 * c.crank;
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t v[32];
                tmem_ld32(c.tmem + kTmemO + lane_base + 32 * cc, v);
                tmem_wait_ld();
                if (h < H) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcg(reinterpret_cast<float4*>(po + 32 * cc + 4 * q),
                               make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
                }
            }
            if (h < H) __stcg(p.ml + (ub * 2 + c.crank) * H + h, make_float2(m_used, lsum));
            __threadfence();
            softmax_bar();
            if (h == 0) {
                const uint32_t old = atomicAdd(p.counters + 2 * r + c.crank, 1u);
                *flag = (old == (uint32_t)(d.s_r - 1)) ? 1u : 0u;
            }
            softmax_bar();
            if (*flag != 0u) {
                __threadfence();
                if (h < H) {
                    float M = sink2;
                    for (int i = 0; i < d.s_r; ++i)
                        M = fmaxf(M, __ldcg(p.ml + ((size_t)(d.row_u0 + i) * 2 + c.crank) * H + h).x);
                    float Z = 0.f, lall = 0.f;
                    if (M != -INFINITY) {
                        Z = (sink2 == -INFINITY) ? 0.f : exp2f(sink2 - M);
                        for (int i = 0; i < d.s_r; ++i) {
                            const float2 ml = __ldcg(p.ml + ((size_t)(d.row_u0 + i) * 2 + c.crank) * H + h);
                            if (ml.x != -INFINITY) Z += ml.y * exp2f(ml.x - M);
                            lall += ml.y;
                        }
                    }
                    const float inv = Z > 0.f ? 1.f / Z : 0.f;
                    uint16_t* outp = static_cast<uint16_t*>(a.out) + ((size_t)r * H + h) * SMLA_HEAD_DIM + 256 * c.crank;
#pragma unroll 1
                    for (int cc = 0; cc < 8; ++cc) {
                        float acc[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
                        for (int i = 0; i < d.s_r; ++i) {
                            const size_t u = (size_t)(d.row_u0 + i);
                            const float mi = __ldcg(p.ml + (u * 2 + c.crank) * H + h).x;
                            if (mi == -INFINITY) continue;
                            const float w = exp2f(mi - M) * inv;
                            const float* src = p.po + (u * H + h) * SMLA_HEAD_DIM + 256 * c.crank + 32 * cc;
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
                            *reinterpret_cast<uint4*>(outp + 32 * cc + 8 * q) = wv;
                        }
                    }
                    if (c.crank == 0 && a.lse != nullptr) {
                        float lse = (M == -INFINITY || Z <= 0.f) ? -INFINITY : (M + log2f(Z)) * kLn2;
                        if (lall == 0.f) lse = a.sink != nullptr ? __ldg(a.sink + h) : -INFINITY;  // sink only, exactly
                        a.lse[(size_t)r * H + h] = lse;
                    }
                }
                if (h == 0) atomicExch(p.counters + 2 * r + c.crank, 0u);
            }
        }
        // All TMEM reads of O are complete (tcgen05.wait::ld) before the next
        // unit's Q is staged; its first PV (which overwrites O) waits for Q.
        tc_fence_before();
        softmax_bar();
    }
    if (!ok) err |= SMLA_DEV_TIMEOUT;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
smla_decode_kernel(const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const smla_decode_args& a = p.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx c;
    c.sb = smem_addr(smem);
    c.crank = cluster_ctarank();
    c.peer = c.crank ^ 1u;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc);
    c.abort = misc + 1;
    long long* red = reinterpret_cast<long long*>(smem + kOffMisc + 64);
    int* s_tiles = reinterpret_cast<int*>(smem + kOffSin);
    int* s_prefix = s_tiles + SMLA_MAX_ROWS;
    UnitDesc* units = reinterpret_cast<UnitDesc*>(smem + kOffUnits);
    const int R = a.num_rows;
    const int cluster = blockIdx.x >> 1;
    const int n_clusters = gridDim.x >> 1;

    uint32_t err = 0;
    if (tid == 0) {
        misc[1] = 0u;
        mbar_init(bar_addr(c, BAR_Q_READY), kSoftmaxWarps);
        for (int i = 0; i < kNR; ++i) {
            mbar_init(bar_addr(c, BAR_RAW_FULL + i), 1);
            mbar_init(bar_addr(c, BAR_RAW_EMPTY + i), kNumDequantWarps);
        }
        for (int i = 0; i < kNX; ++i) {
            mbar_init(bar_addr(c, BAR_X_FULL + i), kNumDequantWarps);
            mbar_init(bar_addr(c, BAR_X_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_addr(c, BAR_S_FULL + i), 1);
            mbar_init(bar_addr(c, BAR_P_FULL + i), kSoftmaxWarps);
        }
        mbar_init(bar_addr(c, BAR_O_DONE), 1);
        mbar_init(bar_addr(c, BAR_EX_FULL), kHeadsPad);
        mbar_init(bar_addr(c, BAR_EX_EMPTY), kHeadsPad);
        mbar_init(bar_addr(c, BAR_MMA_FINAL), 1);
        fence_mbar_init_cluster();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(c.sb + kOffMisc, kTmemCols);
        tmem_relinquish();
    }

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
    if (lane == 0) red[16 + warp] = local_max;
    __syncthreads();
    int max_t = 1;
    for (int w = 0; w < kWarps; ++w) max_t = max(max_t, (int)red[16 + w]);
    int lo = 1, hi = max_t;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        long long cnt = 0;
        for (int r = tid; r < R; r += kThreads) cnt += max(1, ceil_div_i(s_tiles[r], mid));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        __syncthreads();
        if (lane == 0) red[warp] = cnt;
        __syncthreads();
        long long tot = 0;
        for (int w = 0; w < kWarps; ++w) tot += red[w];
        if (tot <= p.units) hi = mid; else lo = mid + 1;
    }
    const int chunk = lo;
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
    // this cluster's units: cluster, cluster + n_clusters, ...
    if (tid == 0) {
        int n = 0;
        for (int u = cluster; u < total_units && n < kMaxUnitsPerCluster; u += n_clusters, ++n) {
            int l2 = 0, h2 = R - 1;  // last r with prefix[r] <= u
            while (l2 < h2) {
                const int mid = (l2 + h2 + 1) >> 1;
                if (s_prefix[mid] <= u) l2 = mid; else h2 = mid - 1;
            }
            UnitDesc d;
            d.row = l2;
            d.row_u0 = s_prefix[l2];
            d.s_r = s_prefix[l2 + 1] - d.row_u0;
            d.unit = u;
            const int T = s_tiles[l2];
            const int tps = T > 0 ? ceil_div_i(T, d.s_r) : 0;
            d.t_begin = min(T, (u - d.row_u0) * tps);
            d.t_end = min(T, d.t_begin + tps);
            d.pad0 = d.pad1 = 0;
            units[n] = d;
        }
        misc[2] = (uint32_t)n;
    }
    if (blockIdx.x == 0 && plan_err) err |= plan_err;
    tc_fence_before();
    cluster_sync();  // barrier inits visible to the peer; plan scratch no longer needed
    tc_fence_after();
    c.tmem = misc[0];
    const int n_units = (int)misc[2];

    if (warp < kSoftmaxWarps) {
        softmax_role(p, c, units, n_units, err);
    } else if (warp < kProducerWarp0 + kNumProducers) {
        producer_role(p, c, units, n_units, warp - kProducerWarp0, err);
        if (c.crank != 0) err &= ~(SMLA_DEV_BAD_INDEX | SMLA_DEV_BAD_CMP);  // reported once, by CTA 0
    } else if (warp == kMmaWarp) {
        if (lane == 0) mma_role(c, units, n_units);
        __syncwarp();
    } else {
        dequant_role(c, units, n_units, warp - kDequantWarp0);
    }

    if (*c.abort) err |= SMLA_DEV_TIMEOUT;
    if (err != 0u) atomicOr(p.err, err);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(c.tmem, kTmemCols);
    }
    cluster_sync();
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
namespace {
std::atomic<int> g_attr_done[64];
std::atomic<int> g_num_sms[64];  // co-resident CTA pairs per device
std::mutex g_attr_mu;

cudaError_t ensure_kernel_attrs(int dev) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_attr_done[dev].load(std::memory_order_acquire) == 1) return cudaSuccess;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (g_attr_done[dev].load(std::memory_order_relaxed) == 1) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(smla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    // co-resident CTA pairs of this kernel (cluster placement follows the GPC layout)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int pairs = 0;
    e = cudaOccupancyMaxActiveClusters(&pairs, smla_decode_kernel, &cfg);
    if (e != cudaSuccess || pairs < 1) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        pairs = sms / 2;
    }
    g_num_sms[dev].store(pairs, std::memory_order_relaxed);
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
    // Persistent grid: one CTA pair per two SMs, at most one pair per unit, and
    // enough pairs that none is handed more than kMaxUnitsPerCluster units.
    const int pairs_resident = std::max(1, g_num_sms[dev].load(std::memory_order_relaxed));
    int clusters = std::min(kp.units, pairs_resident);
    clusters = std::max(clusters, (kp.units + kMaxUnitsPerCluster - 1) / kMaxUnitsPerCluster);
    const dim3 grid((unsigned)(2 * clusters)), block(kThreads);
    smla_decode_kernel<<<grid, block, kSmemBytes, stream>>>(kp);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
