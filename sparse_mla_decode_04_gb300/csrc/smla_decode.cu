// Sparse-MLA decode for sm_103a: kernel and launch.
//
// Method ("[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on gfx950",
// section "Design"): per query row, one 512-wide QK dot (448 NoPE + 64 RoPE
// dims) against the entries the row selects (top-k main-cache slots with -1 as
// an invalid slot, a sliding window, compressed-cache 64-entry groups with a
// masked tail), a softmax with a per-head sink logit, and a 512-wide PV.
// Split plan, merge of split rows and graph safety follow "[ASM] [HIP] [MLA v4
// nm] Split plan helper and persistent decode kernel with in-kernel split and
// merge", summary part 2 (here the merge is a second, GPU-wide kernel).
//
// GB300 design.  A work unit is (row, split).  O for 128 heads x 512 dims in
// fp32 would fill a whole SM's TMEM, so each unit runs on two CTAs and CTA c
// owns output dims [256c, 256c+256).  The two CTAs share nothing: each one
// gathers the whole entries and computes the full 512-wide QK itself, so both
// hold bit-identical scores and make identical softmax decisions, and no data
// crosses SMs (moving partial scores between SMs through distributed shared
// memory measured ~2.5 us per 32 KB, several times the tensor time of a tile).
// The grid is persistent.  Inside a CTA, warp roles pass tiles along
// mbarrier rings.  A tile is 64 entries (the N of QK: a tcgen05 MMA with
// M = 128 costs about the same for N = 32 and N = 64, so 64 halves the QK
// cost per entry); entries are fetched in 32-entry raw tiles, two per tile.
//
//   producer warps (3)   one per raw stage: resolve a raw tile's 32 slots (top-k index -> page
//                        table -> 64-bit row; window; compressed) and fetch the
//                        valid entries (576 B each) into a 3-stage raw ring: one
//                        bulk copy for a run of consecutive pool rows, else
//                        16-byte cp.async gathers; plus a cp.async of each
//                        entry's 8 scale bytes;
//   dequant warps (8)    raw ring -> bf16 (e4m3 x 2^(code-127), exact) in
//                        128-byte-swizzled [4 atoms][64][128 B] halves of a
//                        tile: this CTA's 256 dims ("own": the K-major B of QK
//                        and the MN-major B of PV) in a 2-stage ring, the other
//                        256 dims ("peer": QK only) in a single stage that is
//                        refilled as soon as QK of the previous tile is done;
//   MMA warp (1 thread)  QK(t): M = 128 heads, N = 64, K = 512 with Q's peer
//                        dims from TMEM and its own dims from shared memory;
//                        then PV(t-1): M = 128, N = 256, K = 64 with P from TMEM;
//                        the issue rate of this one thread bounds the tile;
//   softmax warps (4)    one thread per head (TMEM lane): online softmax with a
//                        conditional rescale, P written back over the scores as
//                        a bf16 pair hi = bf16(p), lo = bf16(p - hi).  A single
//                        bf16 P (8-bit mantissa) is not enough: with V near 600
//                        in magnitude, nearly tied entries whose V values cancel
//                        would carry errors near 1.  The lo half is skipped on
//                        tiles where a running bound (sum |lo| x max |V|) shows
//                        its total effect on every head's output stays within
//                        2^-9; on peaked softmaxes most tiles qualify.
//
// TMEM (512 columns): O [0, 256), two score/P buffers [256, 320) and
// [320, 384), Q's peer dims (the 256 this CTA does not output) as bf16 pairs
// [384, 512).  Heads beyond num_heads are zero-padded up to the MMA's M = 128.
//
// Split rows leave fp32 partials; a second launch (smla_merge_kernel, one
// block per row, dim half and 8 heads) combines them over the whole GPU.
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

constexpr int kBK = 64;               // entries per tile (QK N, PV K)
constexpr int kRawBK = 32;            // entries per raw tile (one producer lane each)
constexpr int kRawPerTile = kBK / kRawBK;
constexpr int kNR = 3;                // raw-byte ring stages
constexpr int kNXO = 2;               // own-dims tile stages
// Softmax warps 0-7: warp w serves heads 32 (w % 4) .. 32 (w % 4) + 31 (TMEM
// lanes, one thread per head) and side w / 4 of each tile: entries
// 32 (w / 4) .. 32 (w / 4) + 31.  Side 0 also stages Q and finishes units.
constexpr int kSoftmaxWarps = 8;
constexpr int kSideWarps = 4;
constexpr int kProducerWarp0 = 8;     // warps 8-10: producer pw owns raw stage pw (tiles g % kNR == pw)
constexpr int kNumProducers = kNR;    // one per stage: each waits its stage's phases strictly in order
constexpr int kMmaWarp = 11;
constexpr int kDequantWarp0 = 12;     // warps 12-19
constexpr int kNumDequantWarps = 8;
constexpr int kWarps = 20;
constexpr int kThreads = 32 * kWarps;
constexpr int kHeadsPad = 128;        // heads padded up to the MMA M
static_assert(kHeadsPad == 32 * kSideWarps, "one softmax thread per padded head on each side");
static_assert(kRawBK == 32, "one producer lane per slot");
constexpr int kMaxUnitsPerPair = 32;
constexpr int kUnitCostTiles = 2;     // plan estimate: staging + finishing a unit, in tiles
constexpr int kMinStreamTiles = 4;    // a stream-plan range is at least this many tiles
constexpr int kMaxStreamRanges = 96;  // stream-plan ranges (pairs) at most: bounds a row's partials
constexpr int kPlanWarp = 1;          // computes the split plan during setup

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;        // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;      // score / P buffers: [256, 320), [320, 384)
constexpr uint32_t kTmemQ = 384;      // Q's peer dims, bf16 packed: [384, 512)
constexpr uint64_t kDrainNs = 2000000000ull;  // limit of the teardown waits for work already issued (2 s)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// log2 units: P may grow to 2^32 before O is rescaled.  O then stays below
// n * 2^32 * max|x|, far inside fp32's range for any row length and scale
// codes up to about 190, and the (TMEM-heavy) rescale of O becomes rare.
constexpr float kRescaleThreshold = 32.0f;
// The lo half of P is skipped on a tile only while, for every head, the bound
// on everything skipped so far stays within kLoBudget of the running softmax
// denominator: the output error from skipping is then at most kLoBudget.
constexpr float kLoBudget = 1.0f / 512.0f;

constexpr uint32_t kAtomBytes = kBK * 128;                      // one 64-dim atom of a tile: 8 KB
constexpr uint32_t kHalfBytes = 4 * kAtomBytes;                 // 256 dims of a tile: 32 KB
constexpr uint32_t kRawStageBytes = kRawBK * SMLA_ENTRY_BYTES;  // 18 KB

// Shared-memory layout (offsets from a 1024-byte-aligned base).
constexpr uint32_t kOffQ = 0;                                      // Q's own dims: [4 atoms][128][128 B]
constexpr uint32_t kOffXO = kOffQ + 65536;                         // own dims: [kNXO][4 atoms][64][128 B]
constexpr uint32_t kOffXP = kOffXO + kNXO * kHalfBytes;            // peer dims: [4 atoms][64][128 B]
constexpr uint32_t kOffRaw = kOffXP + kHalfBytes;                  // [kNR][32][576 B]
constexpr uint32_t kOffRawSc = kOffRaw + kNR * kRawStageBytes;     // [kNR][32] u64 scale codes
constexpr uint32_t kOffRawMask = kOffRawSc + kNR * kRawBK * 8;     // [kNR][4] u32: loaded, valid for A, for B
constexpr uint32_t kOffXMask = kOffRawMask + kNR * 16;             // [kNXO][2 raw tiles][A, B] u32 valid masks
constexpr uint32_t kOffXVmax = kOffXMask + kNXO * 16;              // [kNXO][8 dequant warps] f32 max |V| bound
constexpr uint32_t kOffXPoison = kOffXVmax + kNXO * 32;            // [kNXO][8 dequant warps] u32 rows poisoned (bit 0 A, 1 B)
constexpr uint32_t kOffVote = kOffXPoison + kNXO * 32;             // [2][4 head quarters] u32 lo-skip votes
constexpr uint32_t kOffXch = kOffVote + 32;                        // [3][2 sides][128 heads] f32 side exchange
constexpr uint32_t kOffBar = kOffXch + 3 * 2 * 128 * 4;         // mbarriers
constexpr uint32_t kNumBars = 32;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;           // tmem base, flags, reductions
constexpr uint32_t kMiscBytes = 512;
constexpr uint32_t kOffUnits = kOffMisc + kMiscBytes;           // unit descriptors
constexpr uint32_t kSmemUsed = kOffUnits + kMaxUnitsPerPair * 32;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;               // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
// The plan's per-row scratch (tiles[R], prefix[R+1]) aliases the raw ring
// during the prologue, before any producer runs.
static_assert(4 * (3 * SMLA_MAX_ROWS + 2 * kMaxStreamRanges + 8) <= kNR * kRawStageBytes, "plan scratch fits in the raw ring");

// mbarrier indices
enum : uint32_t {
    BAR_RAW_FULL = 0,                      // [kNR] producer -> dequant (32 async + 1 arrival, tx bytes)
    BAR_RAW_EMPTY = BAR_RAW_FULL + kNR,    // [kNR] dequant -> producer (kNumDequantWarps)
    BAR_X_FULL = BAR_RAW_EMPTY + kNR,      // [kNXO] own dims written: dequant -> MMA, softmax (kNumDequantWarps)
    BAR_XP_FULL = BAR_X_FULL + kNXO,       // peer dims written: dequant -> MMA (kNumDequantWarps)
    BAR_XO_EMPTY = BAR_XP_FULL + 1,        // [kNXO] MMA commit after PV (own dims free)
    BAR_XP_EMPTY = BAR_XO_EMPTY + kNXO,    // MMA commit after QK (peer dims free)
    BAR_S_FULL = BAR_XP_EMPTY + 1,         // [2] MMA commit after QK's own-dims half
    BAR_S_PEER = BAR_S_FULL + 2,           // [2] MMA commit after QK's peer-dims half
    BAR_S_PEER_READ = BAR_S_PEER + 2,      // [2] softmax holds the peer partial: its columns are free (kSoftmaxWarps)
    BAR_P_FULL = BAR_S_PEER_READ + 2,      // [2] softmax -> MMA (kSoftmaxWarps)
    BAR_O_DONE = BAR_P_FULL + 2,           // [2] MMA commit after PV(j), on barrier j % 2
    BAR_Q_READY = BAR_O_DONE + 2,          // side-0 softmax -> MMA, once per unit (kSideWarps)
    BAR_MMA_FINAL = BAR_Q_READY + 1,       // teardown: all MMAs retired
    BAR_COUNT = BAR_MMA_FINAL + 1
};
static_assert(BAR_COUNT <= kNumBars, "barrier slots");

struct KParams {
    smla_decode_args a;
    uint32_t* err;
    int2* row_table;     // [SMLA_MAX_ROWS] (first unit, partials) per row: block 0's plan -> merge kernel
    float2* ml;          // [units][2][H]   (m in log2 units, l)
    float* po;           // [units][2][H][256] unnormalised fp32 O, by dims half
    int units;           // num_rows * num_splits: the chunked plan's unit budget
    int unit_cap;        // partial slots in the workspace (>= units and >= rows + kMaxPairs - 1)
    uint64_t wait_ns;    // limit of every pipeline wait (smla_set_wait_limit_ns; default 2 s)
    int pair;            // 1: rows 2v and 2v+1 share a work row (num_heads <= 64), else 0
    int vrows;           // work rows: ceil(num_rows / 2) when paired, else num_rows
    int lanes;           // heads of a partial (its stride): 128 when paired, else num_heads
};

struct UnitDesc {
    int row, s_r, row_u0, unit, t_begin, t_end;
    int pad0, pad1;
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

// The same conversion by bit placement.  Moving an e4m3 code's 7 magnitude
// bits to bf16 bits 4..10 and its sign to bit 15 gives a bf16 that reads
// exactly 2^-120 times the e4m3 value (normal codes land on normal bf16
// numbers, subnormal codes on bf16 subnormals with the same factor).  One
// bf16x2 multiply by 2^(code - 7) then yields e4m3 x 2^(code - 127) exactly
// whenever the product is a normal bf16: scale codes 10..134.  A NaN byte
// (magnitude 0x7F) comes out as the finite 480 x 2^(code - 127), above the
// largest e4m3 value 448; fast_chunk_bad() flags both cases.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Elementwise max of |a|, |b| (the sign of the result is not used).
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ void dequant16_fast(const uint4 raw, uint32_t code, uint32_t (&o)[8]) {
    const uint32_t scale2 = ((code + 120u) << 7) * 0x00010001u;  // bf16x2 of 2^(code - 7)
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bytes 0,1 (then 2,3), each followed by a byte of copies of its sign bit
        const uint32_t lo = prmt(w[i], 0x9180u), hi = prmt(w[i], 0xB3A2u);
        o[2 * i] = mul_bf16x2((lo << 4) & 0x87F087F0u, scale2);
        o[2 * i + 1] = mul_bf16x2((hi << 4) & 0x87F087F0u, scale2);
    }
}
// Largest |x| over 8 packed bf16 words, as the 15 magnitude bits of a bf16.
__device__ __forceinline__ uint32_t absmax_bits8(const uint32_t (&o)[8]) {
    const uint32_t m = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(o[0], o[1]), max_abs_bf16x2(o[2], o[3])),
                                      max_abs_bf16x2(max_abs_bf16x2(o[4], o[5]), max_abs_bf16x2(o[6], o[7])));
    return max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
}
// True when dequant16_fast's output for this chunk is not the exact one: a
// scale code outside 10..134, or a NaN byte (a magnitude above 448 x scale).
__device__ __forceinline__ bool fast_chunk_bad(uint32_t code, uint32_t amax_bits) {
    return code - 10u > 124u || amax_bits > (((code + 8u) << 7) | 0x60u);
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

// A work row.  With num_heads <= 64 two rows share one: rows A = 2v and
// B = 2v + 1 (B absent when num_rows is odd) take TMEM lanes [0, 64) and
// [64, 128), and the MMA's M = 128 is filled by both.  Its slots, each
// segment padded to 32-entry raw tiles:
//   A's top-k slots; B's top-k slots;
//   the window: the union of A's and B's windows when both read the same
//     sequence, else A's window then B's;
//   the compressed entries: the union when both start at the same compressed
//     row, else A's then B's.
// Each slot is valid for A, for B or both (a position inside both windows, a
// compressed entry below both lengths).  Without pairing the work row is the
// row itself (B absent) and its slots are exactly the row's.  Two rows of a
// multi-token decode of one sequence share nearly all of their window and
// compressed entries, which are then gathered and multiplied once.
struct VRow {
    int rA, rB;             // rows (rB = -1: absent)
    int seqA, seqB;
    int nmt;                // raw tiles of one row's top-k
    int wsA, wlA, wsB, wlB; // windows: start and length per row
    int w0, wn;             // the union window (wu)
    long long csA, csB;     // compressed: first row per row
    int clA, clB, cn;       // lengths, and the union's (cu)
    bool wu, cu;
    int nA, nB, nW, nC;     // raw tiles of the four segments
};

__device__ __forceinline__ VRow make_vrow(const KParams& p, int v, uint32_t& err) {
    const smla_decode_args& a = p.a;
    VRow w;
    w.rA = p.pair ? 2 * v : v;
    w.rB = (p.pair && 2 * v + 1 < a.num_rows) ? 2 * v + 1 : -1;
    w.seqA = a.row_seq != nullptr ? __ldg(a.row_seq + w.rA) : w.rA;
    w.seqB = w.rB < 0 ? -1 : (a.row_seq != nullptr ? __ldg(a.row_seq + w.rB) : w.rB);
    w.nmt = ceil_div_i(a.topk, kRawBK);
    auto win = [&](int r, int& st, int& ln) {
        st = 0; ln = 0;
        if (r < 0 || a.swa_len == nullptr) return;
        ln = __ldg(a.swa_len + r);
        if (ln < 0) { err |= SMLA_DEV_BAD_LENGTH; ln = 0; }
        st = __ldg(a.swa_start + r);
    };
    auto cmpr = [&](int r, long long& st, int& ln) {
        st = 0; ln = 0;
        if (r < 0 || a.cmp_len == nullptr) return;
        ln = __ldg(a.cmp_len + r);
        if (ln < 0) { err |= SMLA_DEV_BAD_LENGTH; ln = 0; }
        st = __ldg(a.cmp_start + r);
    };
    win(w.rA, w.wsA, w.wlA);
    win(w.rB, w.wsB, w.wlB);
    cmpr(w.rA, w.csA, w.clA);
    cmpr(w.rB, w.csB, w.clB);
    w.wu = w.rB >= 0 && w.seqA == w.seqB && w.wlA > 0 && w.wlB > 0;
    if (w.wu) {
        w.w0 = min(w.wsA, w.wsB);
        w.wn = max(w.wsA + w.wlA, w.wsB + w.wlB) - w.w0;
        // a union longer than the two windows laid end to end saves nothing
        if (w.wn > w.wlA + w.wlB) w.wu = false;
    }
    w.cu = w.rB >= 0 && w.csA == w.csB && w.clA > 0 && w.clB > 0;
    w.cn = w.cu ? max(w.clA, w.clB) : 0;
    w.nA = w.nmt;
    w.nB = w.rB >= 0 ? w.nmt : 0;
    w.nW = w.wu ? ceil_div_i(w.wn, kRawBK) : ceil_div_i(w.wlA, kRawBK) + ceil_div_i(w.wlB, kRawBK);
    w.nC = w.cu ? ceil_div_i(w.cn, kRawBK) : ceil_div_i(w.clA, kRawBK) + ceil_div_i(w.clB, kRawBK);
    return w;
}

// Number of 64-entry tiles of a work row (two raw tiles per tile; the last
// one may be half empty).
__device__ __forceinline__ int vrow_tiles(const VRow& w) { return ceil_div_i(w.nA + w.nB + w.nW + w.nC, kRawPerTile); }

// Slot `lane` of raw tile t of a work row: the pool row (phys >= 0, in the
// compressed pool when *cmp), and for which of A, B it counts.
__device__ __forceinline__ long long vrow_slot(const smla_decode_args& a, const VRow& w, int t, int lane, bool& cmp,
                                               bool& vA, bool& vB, uint32_t& err) {
    long long phys = -1;
    cmp = false;
    vA = vB = false;
    if (t < w.nA + w.nB) {  // top-k of A, then of B
        const bool isB = t >= w.nA;
        const int r = isB ? w.rB : w.rA;
        const int j = (isB ? t - w.nA : t) * kRawBK + lane;
        if (j < a.topk) {
            const int idx = __ldg(a.main_idx + (size_t)r * a.topk + j);
            if (idx != -1) {
                phys = map_position(a, idx, isB ? w.seqB : w.seqA);
                if (phys < 0) err |= SMLA_DEV_BAD_INDEX;
                else { vA = !isB; vB = isB; }
            }
        }
        return phys;
    }
    t -= w.nA + w.nB;
    if (t < w.nW) {  // window
        long long pos;
        int seq;
        if (w.wu) {
            const int j = t * kRawBK + lane;
            if (j >= w.wn) return -1;
            pos = (long long)w.w0 + j;
            vA = pos >= w.wsA && pos < (long long)w.wsA + w.wlA;
            vB = pos >= w.wsB && pos < (long long)w.wsB + w.wlB;
            seq = w.seqA;
        } else {
            const int tA = ceil_div_i(w.wlA, kRawBK);
            const bool isB = t >= tA;
            const int j = (isB ? t - tA : t) * kRawBK + lane;
            if (j >= (isB ? w.wlB : w.wlA)) return -1;
            pos = (long long)(isB ? w.wsB : w.wsA) + j;
            vA = !isB;
            vB = isB;
            seq = isB ? w.seqB : w.seqA;
        }
        phys = map_position(a, pos, seq);
        if (phys < 0) {
            err |= SMLA_DEV_BAD_INDEX;
            vA = vB = false;
        }
        return phys;
    }
    t -= w.nW;
    if (t < w.nC) {  // compressed entries
        long long start;
        int j;
        if (w.cu) {
            j = t * kRawBK + lane;
            if (j >= w.cn) return -1;
            start = w.csA;
            vA = j < w.clA;
            vB = j < w.clB;
        } else {
            const int tA = ceil_div_i(w.clA, kRawBK);
            const bool isB = t >= tA;
            j = (isB ? t - tA : t) * kRawBK + lane;
            if (j >= (isB ? w.clB : w.clA)) return -1;
            start = isB ? w.csB : w.csA;
            vA = !isB;
            vB = isB;
        }
        cmp = true;
        phys = start + j;
        if (phys < 0 || phys >= a.n_cmp) {
            err |= SMLA_DEV_BAD_CMP;
            phys = -1;
            vA = vB = false;
        }
        return phys;
    }
    return -1;
}

// Per-CTA state shared by the roles.
struct Ctx {
    uint32_t sb;              // shared base (1024-aligned)
    uint32_t tmem;            // TMEM base address
    uint32_t half;            // 0 or 1: output dims [256 half, 256 half + 256)
    volatile uint32_t* abort; // set by any role whose bounded wait gave up
    uint64_t wait_ns;         // limit of a pipeline wait
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, uint32_t i) { return c.sb + kOffBar + 8 * i; }

// Bounded wait that also gives up as soon as another role of this CTA aborted.
__device__ __forceinline__ bool wait_bar(const Ctx& c, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        for (int i = 0; i < 4; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if (global_timer_ns() - t0 > c.wait_ns) {
            *c.abort = 1u;
            return false;
        }
    }
}

// The same wait, taken by a whole warp: the outcome is made warp-uniform so
// that the warp never splits around warp-synchronous code after a timeout.
__device__ __forceinline__ bool wait_bar_warp(const Ctx& c, uint32_t bar, uint32_t parity) {
    const bool ok = wait_bar(c, bar, parity);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Named barriers (id 0 is __syncthreads): 1 = all softmax warps, 2..5 = the
// two warps of a head quarter, 6 = the side-0 softmax warps.  Every softmax
// warp runs the same sequence of them (no early exit between two of them),
// so none can be left waiting.
__device__ __forceinline__ void side0_bar() {
    asm volatile("bar.sync 6, %0;" :: "r"(kSideWarps * 32) : "memory");
}

// AND of `v` over the threads of named barrier `id` (`count` threads).
__device__ __forceinline__ bool bar_all(uint32_t id, uint32_t count, bool v) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v), "r"(id), "r"(count) : "memory");
    return r != 0u;
}
// AND over all softmax warps: every softmax thread reaches it once per unit.
__device__ __forceinline__ bool softmax_all(bool v) { return bar_all(1u, kSoftmaxWarps * 32, v); }
// AND over the two warps of head quarter qw (the values of both sides are
// exchanged through shared memory around it).
__device__ __forceinline__ bool pair_all(int qw, bool v) { return bar_all(2u + (uint32_t)qw, 64u, v); }

// ---------------------------------------------------------------------------
// role: producer (warp pw owns raw stage pw: raw tiles q % kNR == pw, where q
// counts this CTA's raw tiles, two per tile; lane = slot).  A parity wait
// cannot tell "two phases ahead" from "previous phase done", so each stage
// has exactly one producer, which waits its phases in order.
// ---------------------------------------------------------------------------
__device__ void producer_role(const KParams& p, const Ctx& c, const UnitDesc* units, int n_units, int pw,
                              uint32_t& err) {
    const smla_decode_args& a = p.a;
    const int lane = threadIdx.x & 31;
    uint32_t q = 0;
    int64_t last_fill = -1;  // the last raw tile this warp filled (all of them go to its stage pw)
    // Nothing this warp started may still be writing shared memory when it
    // leaves, whether it finished or gave up: its cp.async copies are waited
    // for, and so is the phase of its last fill, which completes once the
    // bytes of that fill (bulk or cp.async) have landed.  Only this warp fills
    // its stage, so the barrier cannot have moved past that phase.
    auto drain = [&]() {
        cp_async_wait_all();
        if (last_fill >= 0)
            mbar_wait_bounded(bar_addr(c, BAR_RAW_FULL + (uint32_t)pw), (uint32_t)((last_fill / kNR) & 1), kDrainNs);
        __syncwarp();
    };
    for (int ui = 0; ui < n_units; ++ui) {
        const UnitDesc d = units[ui];
        const VRow w = make_vrow(p, d.row, err);
        for (int t = kRawPerTile * d.t_begin; t < kRawPerTile * d.t_end; ++t, ++q) {
            if ((int)(q % kNR) != pw) continue;
            const uint32_t rs = q % kNR, rph = (q / kNR) & 1u;
            // resolve this lane's slot (raw tiles past the row's end stay empty)
            bool cmp, vA, vB;
            long long phys = vrow_slot(a, w, t, lane, cmp, vA, vB, err);
            if (!(vA || vB)) phys = -1;
            const uint8_t* ep = nullptr;
            const uint8_t* sp = nullptr;
            if (phys >= 0) {
                ep = static_cast<const uint8_t*>(cmp ? a.cmp_pool : a.kv_pool) + phys * SMLA_ENTRY_BYTES;
                sp = static_cast<const uint8_t*>(cmp ? a.cmp_scales : a.kv_scales) + phys * SMLA_SCALE_BYTES;
            }
            const uint32_t mask = __ballot_sync(0xffffffffu, ep != nullptr);
            // A run of consecutive pool rows in lanes 0..n-1 (compressed entries,
            // window entries within a page) moves as one bulk copy.  Other tiles
            // are gathered with 16-byte cp.async (4 lanes per entry, 8 entries
            // per instruction): 36 instructions per lane instead of 32 bulk
            // copies queued on the TMA unit.
            const uint8_t* ep0 = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(ep), 0));
            const int nvalid = __popc(mask);
            const bool run = (mask == (nvalid == 32 ? 0xffffffffu : (1u << nvalid) - 1u)) &&
                             __all_sync(0xffffffffu, ep == nullptr || ep == ep0 + (size_t)lane * SMLA_ENTRY_BYTES);
            // Start the entries' trip from HBM now; the copy into the stage, once
            // the stage is free, then finds them in L2.
            if (run) {
                if (lane == 0 && nvalid > 0) bulk_prefetch_l2(ep0, (uint32_t)nvalid * SMLA_ENTRY_BYTES);
            } else if (ep != nullptr) {
                bulk_prefetch_l2(ep, SMLA_ENTRY_BYTES);
            }
            if (!wait_bar_warp(c, bar_addr(c, BAR_RAW_EMPTY + rs), rph ^ 1u)) { drain(); return; }
            const uint32_t full = bar_addr(c, BAR_RAW_FULL + rs);
            const uint32_t dst = c.sb + kOffRaw + rs * kRawStageBytes;
            if (run) {
                if (lane == 0 && nvalid > 0) {
                    mbar_expect_tx_only(full, (uint32_t)nvalid * SMLA_ENTRY_BYTES);
                    bulk_g2s(dst, ep0, (uint32_t)nvalid * SMLA_ENTRY_BYTES, full);
                }
            } else {
#pragma unroll 1
                for (int rnd = 0; rnd < kRawBK / 8; ++rnd) {
                    const int e = 8 * rnd + (lane >> 2);
                    const uint8_t* src = reinterpret_cast<const uint8_t*>(
                        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(ep), e));
                    if (src != nullptr) {
                        const uint32_t d = dst + (uint32_t)e * SMLA_ENTRY_BYTES;
#pragma unroll
                        for (int j = 0; j < SMLA_ENTRY_BYTES / 64; ++j) {
                            const int k = (lane & 3) + 4 * j;  // 16-byte chunk of the entry
                            cp_async_16(d + 16 * k, src + 16 * k, 16u);
                        }
                    }
                }
            }
            if (ep != nullptr) cp_async_8(c.sb + kOffRawSc + (rs * kRawBK + lane) * 8, sp);
            cp_async_arrive_noinc(full);  // one of the 32 async arrivals
            const uint32_t maskA = p.pair ? __ballot_sync(0xffffffffu, vA && ep != nullptr) : mask;
            const uint32_t maskB = p.pair ? __ballot_sync(0xffffffffu, vB && ep != nullptr) : mask;
            if (lane == 0) {
                st_shared_u32(c.sb + kOffRawMask + rs * 16, mask);
                st_shared_u32(c.sb + kOffRawMask + rs * 16 + 4, maskA);
                st_shared_u32(c.sb + kOffRawMask + rs * 16 + 8, maskB);
                mbar_arrive_local(full);  // the 33rd arrival, ordered after the mask stores
            }
            last_fill = (int64_t)q;
        }
    }
    drain();
}

// ---------------------------------------------------------------------------
// role: dequant (8 warps): raw ring -> bf16 swizzled tile halves
// ---------------------------------------------------------------------------
// A raw tile (32 entries) fills rows [32 k, 32 k + 32) of a tile, k = 0, 1.
// Its dims split in two sets of 4 atoms: set 0 = fp8 dims 0..255 (atoms
// 0..3), set 1 = fp8 dims 256..447 (atoms 4..6) and the bf16 RoPE (atom 7).
// An fp8 warp task is 8 entries x 4 chunks of 16 dims of one atom (lane:
// entry lane/4, chunk lane%4); a RoPE task is 4 entries x 8 chunks (lane:
// entry lane/8, chunk lane%8).  With these shapes every quarter-warp's
// 16-byte raw-ring loads (576-byte entry stride) and swizzled stores fall in 8
// distinct 16-byte bank groups.  Per set and raw tile each warp takes:
//   set 0: fp8 (atom dw/4, entry group dw%4) and (atom 2 + dw/4, group dw%4);
//   set 1: warps 0-3 fp8 (atom 4, group dw) and (atom 6, group dw),
//          warps 4-7 fp8 (atom 5, group dw-4) and RoPE tasks 2(dw-4), 2(dw-4)+1.
// A set is written to the 4-atom buffer `dst` (local atom = atom % 4).
// Returns, when `bound` is set, a bound on |x| over the values written.
// With `bound` (the own dims, which PV reads) a chunk that holds a NaN or an
// infinity, of an entry that only one row of a paired work row selects (maskA
// != maskB there), is stored as zeros: the other row must get exactly 0 from
// an entry it does not select, and 0 x NaN is NaN.  The selecting row is
// reported in *poison (bit 0 row A, bit 1 row B) and its outputs become NaN,
// as that row's own arithmetic would have made them.
__device__ __forceinline__ float dequant_set(uint32_t raw, uint32_t rawsc, uint32_t dst, int row0, uint32_t mask,
                                             uint32_t maskA, uint32_t maskB, int set, int dw, int lane, bool bound,
                                             uint32_t& poison) {
    const int ef = 8 * (dw & 3) + (lane >> 2);  // entry of this warp's fp8 tasks
    const bool fvalid = (mask >> (ef & 31)) & 1u;
    int atom[2];
    if (set == 0) { atom[0] = dw >> 2; atom[1] = 2 + (dw >> 2); }
    else { atom[0] = dw < 4 ? 4 : 5; atom[1] = 6; }
    const bool second_fp8 = set == 0 || dw < 4;
    uint4 v[2];
    uint32_t code[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int k = 4 * atom[it] + (lane & 3);
        v[it] = make_uint4(0u, 0u, 0u, 0u);
        code[it] = 127u;
        if (fvalid && (it == 0 || second_fp8)) {
            v[it] = ld_shared_v4(raw + ef * SMLA_ENTRY_BYTES + 16 * k);
            code[it] = ld_shared_u8(rawsc + ef * 8 + atom[it]);
        }
    }
    const bool has_rope = !second_fp8;
    uint4 rv[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    const int kr = lane & 7;
    int er[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        er[it] = 4 * (2 * (dw - 4) + it) + (lane >> 3);
        if (has_rope && ((mask >> (er[it] & 31)) & 1u))
            rv[it] = ld_shared_v4(raw + er[it] * SMLA_ENTRY_BYTES + SMLA_NOPE_DIMS + 16 * kr);
    }

    // straight-line fast path for every chunk; the rare chunks it gets wrong
    // are redone below with the exact conversion
    uint32_t amax = 0u;
    bool bad[2] = {false, false};
    const int kk = (lane & 3) * 2;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        if (it == 1 && !second_fp8) break;
        uint32_t o[8];
        dequant16_fast(v[it], code[it], o);
        const uint32_t am = absmax_bits8(o);
        bad[it] = fast_chunk_bad(code[it], am);
        amax = max(amax, am);
        const uint32_t d = dst + (atom[it] & 3) * kAtomBytes;
        st_shared_v4(d + sw128_offset(row0 + ef, kk), o[0], o[1], o[2], o[3]);
        st_shared_v4(d + sw128_offset(row0 + ef, kk + 1), o[4], o[5], o[6], o[7]);
    }
    float vbound = __uint_as_float(amax << 16);
    if (has_rope) {
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            uint4 rvv = rv[it];
            if (bound) {
                const float ab = bf16x8_absmax(rvv);
                const uint32_t eb = 1u << (er[it] & 31);
                if (ab == INFINITY && ((maskA ^ maskB) & eb)) {  // non-finite, one row only
                    poison |= (maskA & eb) ? 1u : 2u;
                    rvv = make_uint4(0u, 0u, 0u, 0u);
                } else {
                    vbound = fmaxf(vbound, ab);
                }
            }
            st_shared_v4(dst + 3 * kAtomBytes + sw128_offset(row0 + er[it], kr), rvv.x, rvv.y, rvv.z, rvv.w);
        }
    }
    if (__any_sync(0xffffffffu, bad[0] || bad[1])) {  // rare: one copy of the exact path
#pragma unroll 1
        for (int it = 0; it < 2; ++it) {
            const bool b = it == 0 ? bad[0] : bad[1];
            if (!b) continue;
            const uint4 vv = it == 0 ? v[0] : v[1];
            const uint32_t cd = it == 0 ? code[0] : code[1];
            const float scale = ue8m0_to_f32(cd);
            uint32_t o[8];
            dequant16(vv, scale, o);
            const float bnd = e4m3x16_absmax(vv) * scale;
            const uint32_t eb = 1u << (ef & 31);
            if (bound && !(bnd < INFINITY) && ((maskA ^ maskB) & eb)) {  // non-finite, one row only
                poison |= (maskA & eb) ? 1u : 2u;
#pragma unroll
                for (int z = 0; z < 8; ++z) o[z] = 0u;
            } else {
                vbound = (bnd > vbound || bnd != bnd) ? (bnd != bnd ? INFINITY : bnd) : vbound;
            }
            const uint32_t d = dst + ((it == 0 ? atom[0] : atom[1]) & 3) * kAtomBytes;
            st_shared_v4(d + sw128_offset(row0 + ef, kk), o[0], o[1], o[2], o[3]);
            st_shared_v4(d + sw128_offset(row0 + ef, kk + 1), o[4], o[5], o[6], o[7]);
        }
    }
    return bound ? vbound : 0.f;
}

// Per tile g, four steps with one call site (the role's code stays small in
// the instruction cache): the peer set of raw tile 0 and 1 (once QK(g-1) has
// read the peer buffer), announced on XP_FULL so that QK(g) can start on those
// dims; then the own set of raw tile 0 and 1 (once PV(g-2) has read the own
// stage), each raw stage released after its own set; announced on X_FULL.
__device__ void dequant_role(const Ctx& c, const UnitDesc* units, int n_units, int dw, bool pair) {
    const int lane = threadIdx.x & 31;
    uint32_t g = 0;
    for (int ui = 0; ui < n_units; ++ui) {
        const int n = units[ui].t_end - units[ui].t_begin;
        for (int i = 0; i < n; ++i, ++g) {
            const uint32_t xs = g % kNXO;
            uint32_t mask0 = 0u, mask1 = 0u, mab = 0u;  // mab: this lane's (raw tile, A/B) mask, lanes 0..3
            uint32_t mA[kRawPerTile] = {0u, 0u}, mB[kRawPerTile] = {0u, 0u}, poison = 0u;
            float vbound = 0.f;
#pragma unroll 1
            for (int step = 0; step < 2 * kRawPerTile; ++step) {
                const int k = step & 1;
                const bool own = step >= kRawPerTile;
                const uint32_t q = kRawPerTile * g + k;
                const uint32_t rs = q % kNR;
                if (!own) {
                    if (!wait_bar_warp(c, bar_addr(c, BAR_RAW_FULL + rs), (q / kNR) & 1u)) return;
                    const uint32_t m = ld_shared_u32(c.sb + kOffRawMask + rs * 16);
                    if (k == 0) mask0 = m; else mask1 = m;
                    if ((lane >> 1) == k && lane < 4) mab = ld_shared_u32(c.sb + kOffRawMask + rs * 16 + 4 + 4 * (lane & 1));
                    mA[k] = pair ? ld_shared_u32(c.sb + kOffRawMask + rs * 16 + 4) : m;
                    mB[k] = pair ? ld_shared_u32(c.sb + kOffRawMask + rs * 16 + 8) : m;
                    if (k == 0 && !wait_bar_warp(c, bar_addr(c, BAR_XP_EMPTY), (g & 1u) ^ 1u)) return;
                } else if (k == 0) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_XP_FULL));
                    if (!wait_bar_warp(c, bar_addr(c, BAR_XO_EMPTY + xs), ((g / kNXO) & 1u) ^ 1u)) return;
                }
                const uint32_t dst = own ? c.sb + kOffXO + xs * kHalfBytes : c.sb + kOffXP;
                const int set = own ? (int)c.half : 1 - (int)c.half;
                vbound = fmaxf(vbound, dequant_set(c.sb + kOffRaw + rs * kRawStageBytes, c.sb + kOffRawSc + rs * kRawBK * 8,
                                                   dst, kRawBK * k, k == 0 ? mask0 : mask1, mA[k], mB[k], set, dw, lane,
                                                   own, poison));
                if (own) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_RAW_EMPTY + rs));
                }
            }
            if (dw == 0 && lane < 2 * kRawPerTile) st_shared_u32(c.sb + kOffXMask + (xs * 4 + lane) * 4, mab);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) vbound = fmaxf(vbound, __shfl_xor_sync(0xffffffffu, vbound, o));
            if (lane == 0) st_shared_f32(c.sb + kOffXVmax + (xs * kNumDequantWarps + dw) * 4, vbound);
            if (pair) {  // without pairing both rows are one: nothing is ever zeroed
                poison = __reduce_or_sync(0xffffffffu, poison);
                if (lane == 0) st_shared_u32(c.sb + kOffXPoison + (xs * kNumDequantWarps + dw) * 4, poison);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_X_FULL + xs));
        }
    }
}

// ---------------------------------------------------------------------------
// role: MMA issuer (one thread)
// ---------------------------------------------------------------------------
// PV(j): O += P(j) . X(j) over this CTA's dims, P as the hi then (unless every
// softmax warp voted to skip it) the lo bf16 half, both from TMEM.
__device__ __forceinline__ bool issue_pv(const Ctx& c, uint32_t j, bool first_of_unit) {
    const uint32_t sb = j & 1u, xs = j % kNXO;
    if (!wait_bar(c, bar_addr(c, BAR_P_FULL + sb), (j >> 1) & 1u)) return false;
    tc_fence_after();
    const uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
    const uint64_t bd0 = sdesc_sw128(c.sb + kOffXO + xs * kHalfBytes, kAtomBytes, 1024);
    const uint32_t tp = c.tmem + kTmemS + sb * kBK;
    // P of entries 16 kk .. 16 kk + 15: hi at columns [16 kk, 16 kk + 8), lo in the next 8
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk)  // 16 entries (rows) per step: 2048 B
        mma_bf16_ts(c.tmem + kTmemO, tp + 16 * kk, bd0 + (uint64_t)(kk * 2048 >> 4), idesc_pv,
                    (first_of_unit && kk == 0) ? 0u : 1u);
    uint32_t votes = 1u;
#pragma unroll
    for (int w = 0; w < kSideWarps; ++w) votes &= ld_shared_u32(c.sb + kOffVote + (sb * 4 + w) * 4);
    if (votes == 0u) {  // some head needs the lo half of P on this tile
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ts(c.tmem + kTmemO, tp + 16 * kk + 8, bd0 + (uint64_t)(kk * 2048 >> 4), idesc_pv, 1u);
    }
    mma_commit(bar_addr(c, BAR_XO_EMPTY + xs));
    mma_commit(bar_addr(c, BAR_O_DONE + (j & 1u)));
    return true;
}

// Per tile g: QK(g)'s peer half, then its own half, then PV(g-1).  K = 512
// runs as two separate accumulation chains of 256 dims into the same 64
// columns: the peer dims (Q from TMEM, X from the peer buffer) first; the
// softmax warps take that partial into registers (S_PEER_READ), and the own
// dims (Q and X from shared memory) then start a fresh chain in the same
// columns.  The softmax adds the two partials in fp32.  Two chains of 256
// halve the accumulation error of one chain of 512 (the tensor core's
// accumulation is what bounds the logits' precision), and since fp32
// addition is commutative both CTAs of a pair hold bit-identical scores.
__device__ void mma_role(const Ctx& c, const UnitDesc* units, int n_units) {
    const uint32_t idesc_qk = idesc_bf16_f32(128, kBK, false, false);
    const uint64_t q_desc0 = sdesc_sw128(c.sb + kOffQ, 16, 1024);
    const uint64_t xp_desc0 = sdesc_sw128(c.sb + kOffXP, 16, 1024);
    uint32_t g = 0;
    bool ok = true;
    for (int ui = 0; ui < n_units && ok; ++ui) {
        const int n = units[ui].t_end - units[ui].t_begin;
        if (!wait_bar(c, bar_addr(c, BAR_Q_READY), (uint32_t)ui & 1u)) break;
        tc_fence_after();
        const uint32_t g0 = g;
        for (int i = 0; i < n; ++i, ++g) {
            const uint32_t xs = g % kNXO, sb = g & 1u;
            const uint64_t xo_desc0 = sdesc_sw128(c.sb + kOffXO + xs * kHalfBytes, 16, 1024);
            const uint32_t ts = c.tmem + kTmemS + sb * kBK;
            // peer half: its columns last held P(g-2), read by PV(g-2), issued before this
            if (!wait_bar(c, bar_addr(c, BAR_XP_FULL), g & 1u)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_bf16_ts(ts, c.tmem + kTmemQ + kk * 8,
                            xp_desc0 + (uint64_t)(((kk >> 2) * kAtomBytes + (kk & 3) * 32) >> 4), idesc_qk,
                            kk == 0 ? 0u : 1u);
            mma_commit(bar_addr(c, BAR_XP_EMPTY));
            mma_commit(bar_addr(c, BAR_S_PEER + sb));
            // own half: a fresh chain once the softmax holds the peer partial
            if (!wait_bar(c, bar_addr(c, BAR_S_PEER_READ + sb), (g >> 1) & 1u)) { ok = false; break; }
            if (!wait_bar(c, bar_addr(c, BAR_X_FULL + xs), (g / kNXO) & 1u)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_bf16_ss(ts, q_desc0 + (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                            xo_desc0 + (uint64_t)(((kk >> 2) * kAtomBytes + (kk & 3) * 32) >> 4), idesc_qk,
                            kk == 0 ? 0u : 1u);
            mma_commit(bar_addr(c, BAR_S_FULL + sb));
            if (i > 0 && !issue_pv(c, g - 1, (g - 1) == g0)) { ok = false; break; }
        }
        if (ok && n > 0 && !issue_pv(c, g - 1, (g - 1) == g0)) ok = false;
    }
    // retire every MMA before TMEM is released
    mma_commit(bar_addr(c, BAR_MMA_FINAL));
    mbar_wait_bounded(bar_addr(c, BAR_MMA_FINAL), 0, kDrainNs);
}

// ---------------------------------------------------------------------------
// finish stores through shared memory
// ---------------------------------------------------------------------------
// A unit's result leaves TMEM one row per thread (thread = head); stored
// straight to global memory, each 16-byte store of a warp would touch 32 rows.
// Instead each warp stages its 32 rows of 512 bytes in the Q region (free
// between the unit's last QK and the next unit's Q staging) and writes them
// out one row per instruction, 512 contiguous bytes per warp store.  Row h
// sits at Q + 512 h with its 16-byte chunks XOR-swizzled by h % 32, so both
// the row-wise stores and the column-wise loads stay free of bank conflicts.
__device__ __forceinline__ uint32_t stage_addr(const Ctx& c, int h, int chunk) {
    return c.sb + kOffQ + (uint32_t)h * 512u + (uint32_t)((chunk ^ (h & 31)) * 16);
}
// Write this warp's 32 staged rows: lane h's row (when keep(h)) to dst_row(h)
// (512 bytes).
template <class Keep, class RowPtr>
__device__ __forceinline__ void stage_flush(const Ctx& c, int warp, int lane, Keep keep, RowPtr dst_row) {
    __syncwarp();
#pragma unroll 4
    for (int rr = 0; rr < 32; ++rr) {
        const int h = 32 * warp + rr;
        const uint4 v = ld_shared_v4(stage_addr(c, h, lane));
        if (keep(h)) __stcg(reinterpret_cast<uint4*>(dst_row(h)) + lane, v);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// role: softmax / epilogue (warps 0-3, thread = head = TMEM lane)
// ---------------------------------------------------------------------------
__device__ void softmax_role(const KParams& p, const Ctx& c, UnitDesc* units, int n_units, uint32_t& err) {
    const smla_decode_args& a = p.a;
    const int warp = threadIdx.x >> 5;     // 0..7
    const int lane = threadIdx.x & 31;
    const int qw = warp & 3;               // head quarter (TMEM lanes 32 qw ..)
    const int sd = warp >> 2;              // side: tile entries 32 sd .. 32 sd + 31
    const int h = 32 * qw + lane;          // head (TMEM lane) of this thread
    const int H = a.num_heads;
    const uint32_t lane_base = (uint32_t)(qw * 32) << 16;
    const float qscale = a.sm_scale * kLog2e;
    // Lane -> (row of the work row, head): paired work rows put row A on lanes
    // 0..63 and row B on 64..127; lanes past num_heads are padding.
    const int sub = p.pair ? (h >> 6) : 0;       // 0 = row A, 1 = row B
    const int hr = p.pair ? (h & 63) : h;        // head within its row
    const float sink2 = (a.sink != nullptr && hr < H) ? __ldg(a.sink + hr) * kLog2e : -INFINITY;
    uint32_t g = 0;
    bool ok = true;

    for (int ui = 0; ui < n_units && ok; ++ui) {
        const UnitDesc d = units[ui];
        const int rA = p.pair ? 2 * d.row : d.row;
        const int rB = (p.pair && rA + 1 < a.num_rows) ? rA + 1 : -1;
        const int row_of_sub[2] = {rA, rB};
        const int r = row_of_sub[sub];                  // this lane's row (-1: absent)
        const bool live = hr < H && r >= 0;              // this lane carries a real head
        const int n = d.t_end - d.t_begin;
        // ---- Q of this row (side 0): its peer dims (the 256 this CTA does not
        //      output) -> TMEM [384, 512) as bf16 pairs, its own dims -> shared
        //      memory, K-major with the 128-byte swizzle.  The next unit's q rows
        //      are prefetched into L2 now, a unit ahead.
        if (sd == 0) {
            if (h == 0 && ui + 1 < n_units) {
                const int rn0 = p.pair ? 2 * units[ui + 1].row : units[ui + 1].row;
                const int nr = (p.pair && rn0 + 1 < a.num_rows) ? 2 : 1;  // rows of a work row are adjacent
                const size_t rn = (size_t)rn0 * H;
                bulk_prefetch_l2(static_cast<const uint16_t*>(a.q_nope) + rn * SMLA_NOPE_DIMS,
                                 (uint32_t)(nr * H * SMLA_NOPE_DIMS * 2));
                bulk_prefetch_l2(static_cast<const uint16_t*>(a.q_rope) + rn * SMLA_ROPE_DIMS,
                                 (uint32_t)(nr * H * SMLA_ROPE_DIMS * 2));
            }
            // Q in 16-byte chunks j = dims 8j .. 8j + 7 (NoPE chunks 0..55, RoPE
            // 56..63).  Each warp copies its 32 heads one head per instruction
            // (lane = chunk: coalesced) with cp.async, all 32 in flight.  The
            // peer dims' 32 chunks go to TMEM (the A operand of QK's first half)
            // through a row per head staged in the Q region; then the own dims'
            // 32 chunks go straight to their place in the Q region, K-major with
            // the 128-byte swizzle (after every warp has read its staged rows).
            // Heads beyond num_heads are zero-filled.
            const uint4* qn = static_cast<const uint4*>(a.q_nope);
            const uint4* qr = static_cast<const uint4*>(a.q_rope);
            const int pbase = 32 * (1 - (int)c.half), obase = 32 * (int)c.half;
            // lane hh's (row, head): this warp's 32 lanes all belong to one row
            const int wr = row_of_sub[p.pair ? (warp >> 1) : 0];
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                const int j = (pass == 0 ? pbase : obase) + lane;
#pragma unroll 8
                for (int rr = 0; rr < 32; ++rr) {
                    const int hh = 32 * warp + rr;
                    const int hd = p.pair ? (hh & 63) : hh;
                    const bool real = hd < H && wr >= 0;
                    const size_t qrow = real ? (size_t)wr * H + hd : 0;
                    const uint4* src = j < 56 ? qn + qrow * (SMLA_NOPE_DIMS / 8) + j
                                              : qr + qrow * (SMLA_ROPE_DIMS / 8) + (j - 56);
                    const uint32_t dst = pass == 0 ? stage_addr(c, hh, lane)
                                                   : c.sb + kOffQ + (lane >> 3) * 16384 + sw128_offset(hh, lane & 7);
                    cp_async_16(dst, src, real ? 16u : 0u);
                }
                cp_async_wait_all();
                __syncwarp();
                if (pass == 0) {
#pragma unroll 1
                    for (int hc = 0; hc < 4; ++hc) {  // 64 dims -> 32 TMEM columns
                        uint32_t v[32];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint4 w = ld_shared_v4(stage_addr(c, h, 8 * hc + q));
                            v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
                        }
                        tmem_st32(c.tmem + kTmemQ + lane_base + 32 * hc, v);
                    }
                    side0_bar();  // all staged rows read before the own dims overwrite the region
                }
            }
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_Q_READY));
        }

        float m_used = -INFINITY, lsum = 0.f;
        float skipped = 0.f;  // bound on the lo-half contributions skipped so far (units of lsum)
        bool o_init = false;
        bool poisoned = false;  // an entry this row selects held a NaN / inf stored as zeros (dequant_set)
        // QK's peer-dims partial of this side's 32 columns of the tile about to
        // be processed (see mma_role): taken into registers, which frees the
        // columns for the own-dims chain.
        float peer[32];
        auto take_peer = [&](uint32_t gg) -> bool {
            const uint32_t sb = gg & 1u;
            if (!wait_bar_warp(c, bar_addr(c, BAR_S_PEER + sb), (gg >> 1) & 1u)) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(c.tmem + kTmemS + sb * kBK + lane_base + 32 * sd, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) peer[j] = __uint_as_float(v[j]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_S_PEER_READ + sb));
            return true;
        };
        // Both warps of a head quarter hold the same per-head state (m_used,
        // lsum, skipped), exchanged twice per tile through kOffXch; every warp
        // runs every tile's two exchanges even after a failed wait, so the
        // pair barriers always match.
        const uint32_t xch = c.sb + kOffXch;
        auto xch_addr = [&](int k, int side) { return xch + (uint32_t)((k * 2 + side) * 128 + h) * 4u; };
        if (n > 0 && ok) ok = take_peer(g);
        for (int i = 0; i < n; ++i, ++g) {
            const uint32_t sbuf = g & 1u;
            const uint32_t ts = c.tmem + kTmemS + sbuf * kBK + lane_base + 32 * sd;  // this side's 32 columns
            const uint32_t xs = g % kNXO;
            // The tile's valid mask and |V| bound were written before its X_FULL
            // arrival; X_FULL of this tile cannot have advanced further (its stage
            // is refilled only after PV of this tile, which needs this thread's P).
            if (ok && !wait_bar_warp(c, bar_addr(c, BAR_S_FULL + sbuf), (g >> 1) & 1u)) ok = false;
            if (ok && !wait_bar_warp(c, bar_addr(c, BAR_X_FULL + xs), (g / kNXO) & 1u)) ok = false;
            tc_fence_after();
            // this side's 32 entries, valid for this warp's row (quarters 2, 3
            // hold row B of a paired work row; without pairing both masks agree)
            const uint32_t vm = ld_shared_u32(c.sb + kOffXMask + (xs * 4 + 2 * sd + (qw >> 1)) * 4);
            // pass 1: this side's scores (own-dims chain + peer-dims partial, added
            // in fp32 and written back for pass 2) and their masked maximum (taken
            // over the raw scores: qscale > 0)
            float mts = -INFINITY;
            if (ok) {
                uint32_t v[32];
                tmem_ld32(ts, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + peer[j]);
                tmem_st32(ts, v);
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (vm == 0xffffffffu) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(v[j]));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        mx[j & 3] = fmaxf(mx[j & 3], ((vm >> j) & 1u) ? __uint_as_float(v[j]) : -INFINITY);
                }
                mts = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                tmem_wait_st();  // pass 2 reloads the sums
            }
            st_shared_f32(xch_addr(0, sd), mts);
            ok = pair_all(qw, ok);
            const float mt0 = ld_shared_f32(xch_addr(0, 0)) * qscale, mt1 = ld_shared_f32(xch_addr(0, 1)) * qscale;
            const float mt = fmaxf(mt0, mt1);
            float m_new = m_used;
            if (m_used == -INFINITY || mt > m_used + kRescaleThreshold) m_new = fmaxf(m_used, mt);
            const float alpha = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - m_new);
            // m_new is finite once any slot was valid; invalid slots give 2^-inf = +0
            const float msub = (m_new == -INFINITY) ? 0.f : m_new;
            const bool rescale = o_init && (m_new != m_used);
            m_used = m_new;
            // A cold tile: for every head of this quarter, dropping the tile's
            // whole lo half keeps the skipped total within the budget on the bound
            // alone (p <= 2^(mt_side - m) per entry; p - bf16(p) is at most 2^-8 p,
            // bf16's unit roundoff with 8 significant bits, and the stored lo at
            // most (1 + 2^-8) times that; the new denominator is at least
            // lsum alpha).  Then lo is not computed: it is stored as 0 and that
            // bound stands in for its sum.  Both sides take the same decision from
            // the same values.
            const uint32_t vb = c.sb + kOffXVmax + xs * (4 * kNumDequantWarps);
            float vmax = ld_shared_f32(vb);
#pragma unroll
            for (int w = 1; w < kNumDequantWarps; ++w) vmax = fmaxf(vmax, ld_shared_f32(vb + 4 * w));
            if (p.pair) {
                uint32_t pois = 0u;
#pragma unroll
                for (int w = 0; w < kNumDequantWarps; ++w)
                    pois |= ld_shared_u32(c.sb + kOffXPoison + (xs * kNumDequantWarps + w) * 4);
                if (ok && ((pois >> sub) & 1u)) poisoned = true;
            }
            const float capk = 32.f * (1.0f / 256.0f) * (1.0f + 1.0f / 256.0f);
            const float cap0 = mt0 == -INFINITY ? 0.f : capk * ex2_approx(mt0 - msub);
            const float cap1 = mt1 == -INFINITY ? 0.f : capk * ex2_approx(mt1 - msub);
            const bool cold = __all_sync(0xffffffffu, !live || (skipped * alpha + (cap0 + cap1) * vmax <= kLoBudget * lsum * alpha));
            // The next tile's peer partial is taken now (this tile's scores are
            // back in TMEM), so that QK's own-dims chain of the next tile runs
            // while this tile's P is computed.
            if (ok && i + 1 < n) ok = take_peer(g + 1);
            // ---- pass 2: P = 2^(s - m) as a bf16 pair hi = bf16(p), lo = bf16(p - hi),
            // written over this side's columns one 16-entry step at a time:
            // entries 16 q .. 16 q + 15 become hi in columns [16 q, 16 q + 8) and
            // lo in [16 q + 8, 16 q + 16).  Safe before PV(g-1) completes: these
            // columns were last read by PV(g-2), which retired before QK(g) (same
            // issue stream) produced this tile's scores.
            float ps_side = 0.f, lo_side = 0.f;
            if (ok) {
                // pairs of entries in packed fp32x2 arithmetic (each lane of it
                // rounds as the scalar operation would)
                const uint64_t qs2 = f2_pack(qscale, qscale), nm2 = f2_pack(-msub, -msub);
                uint64_t sm2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)}, la2[2] = {sm2[0], sm2[0]};
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    uint32_t v[16];
                    tmem_ld16(ts + 16 * q, v);
                    tmem_wait_ld();
                    const uint32_t vq = (vm >> (16 * q)) & 0xFFFFu;
                    uint32_t hl[16];  // hi pairs, then lo pairs
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), qs2, nm2), x0,
                                  x1);
                        if (vq != 0xFFFFu) {
                            x0 = ((vq >> (2 * j)) & 1u) ? x0 : -INFINITY;
                            x1 = ((vq >> (2 * j + 1)) & 1u) ? x1 : -INFINITY;
                        }
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        const uint64_t p2 = f2_pack(p0, p1);
                        sm2[j & 1] = f2_add(sm2[j & 1], p2);
                        const __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                        memcpy(&hl[j], &hb, 4);
                        if (cold) {
                            hl[8 + j] = 0u;
                        } else {
                            const uint64_t r2 = f2_sub(p2, f2_pack(__low2float(hb), __high2float(hb)));
                            float r0, r1;
                            f2_unpack(r2, r0, r1);
                            hl[8 + j] = pack_bf16(r0, r1);
                            la2[j & 1] = f2_add(la2[j & 1], f2_pack(fabsf(r0), fabsf(r1)));
                        }
                    }
                    tmem_st16(ts + 16 * q, hl);
                }
                float a0, a1, b0, b1;
                f2_unpack(f2_add(sm2[0], sm2[1]), a0, a1);
                ps_side = a0 + a1;
                f2_unpack(f2_add(la2[0], la2[1]), b0, b1);
                // |bf16(r)| <= |r| (1 + 2^-8): a bound on the sum of |lo|
                lo_side = cold ? (sd == 0 ? cap0 : cap1) : (b0 + b1) * (1.0f + 1.0f / 256.0f);
            }
            st_shared_f32(xch_addr(1, sd), ps_side);
            st_shared_f32(xch_addr(2, sd), lo_side);
            ok = pair_all(qw, ok);
            const float ps = ld_shared_f32(xch_addr(1, 0)) + ld_shared_f32(xch_addr(1, 1));
            const float lo_abs = ld_shared_f32(xch_addr(2, 0)) + ld_shared_f32(xch_addr(2, 1));
            lsum = lsum * alpha + ps;
            skipped *= alpha;
            // PV(g-1) must be done before O is rescaled; without a rescale this
            // warp does not wait for it.  Every tile has one PV, PV(j) commits to
            // O_DONE[j % 2], and S_FULL(g) (QK(g) retired, issued after PV(g-2))
            // means PV(g-3) has retired: the barrier is at most one phase behind
            // the one waited for, so a parity wait cannot alias.  Side sd
            // rescales O columns [128 sd, 128 sd + 128).
            const bool need_o = __any_sync(0xffffffffu, rescale);
            if (ok && need_o) {
                if (!wait_bar_warp(c, bar_addr(c, BAR_O_DONE + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u)) ok = false;
                tc_fence_after();
                if (ok) {
                    const float f = rescale ? alpha : 1.f;
#pragma unroll 1
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint32_t oa = c.tmem + kTmemO + lane_base + 128 * sd + 32 * cc;
                        uint32_t v[32];
                        tmem_ld32(oa, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * f);
                        tmem_st32(oa, v);
                    }
                }
            }
            // vote on skipping the lo half: sum|lo| x max|V| (this CTA's dims)
            // bounds what skipping drops; both sides reach the same vote
            {
                const float cand = skipped + lo_abs * vmax;
                const bool mine = !live || cold || (cand <= kLoBudget * lsum);
                const bool warp_ok = __all_sync(0xffffffffu, mine);
                if (warp_ok) skipped = cand;  // counted even if another quarter vetoes: conservative
                if (sd == 0 && lane == 0) st_shared_u32(c.sb + kOffVote + (sbuf * 4 + qw) * 4, warp_ok ? 1u : 0u);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar_addr(c, BAR_P_FULL + sbuf));
            o_init = true;
        }
        if (ok && n > 0) {  // the unit's last PV (PV(g-1)); earlier ones retired before it
            if (!wait_bar_warp(c, bar_addr(c, BAR_O_DONE + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u)) ok = false;
            tc_fence_after();
        }
        if (!softmax_all(ok)) {  // uniform over the softmax warps from here on
            ok = false;
            *c.abort = 1u;
            break;
        }
        if (sd != 0) continue;  // side 0 finishes the unit and stages the next Q
        tc_fence_after();       // side 1's rescales of O are complete (before the barrier)
        if (poisoned) { m_used = NAN; lsum = NAN; }  // the row's partial or outputs become NaN, as a selected NaN makes them
        // ---- finish: final bf16 output, or an fp32 partial for the merge kernel ----
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
            if (lsum == 0.f) lse = (a.sink != nullptr && hr < H) ? __ldg(a.sink + hr) : -INFINITY;  // sink only, exactly
            if (poisoned) { oscale = NAN; lse = NAN; }
            // 256 bf16 dims per head = one 512-byte staged row
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
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_shared_v4(stage_addr(c, h, 4 * cc + q),
                                 pack_bf16(__uint_as_float(v[8 * q]) * oscale, __uint_as_float(v[8 * q + 1]) * oscale),
                                 pack_bf16(__uint_as_float(v[8 * q + 2]) * oscale, __uint_as_float(v[8 * q + 3]) * oscale),
                                 pack_bf16(__uint_as_float(v[8 * q + 4]) * oscale, __uint_as_float(v[8 * q + 5]) * oscale),
                                 pack_bf16(__uint_as_float(v[8 * q + 6]) * oscale, __uint_as_float(v[8 * q + 7]) * oscale));
            }
            {
                const int wr = row_of_sub[p.pair ? (warp >> 1) : 0];  // the row of this warp's 32 lanes
                stage_flush(c, warp, lane, [&](int hh) { return (p.pair ? (hh & 63) : hh) < H && wr >= 0; },
                            [&](int hh) {
                                return static_cast<uint16_t*>(a.out) +
                                       ((size_t)wr * H + (p.pair ? (hh & 63) : hh)) * SMLA_HEAD_DIM + 256 * c.half;
                            });
            }
            if (c.half == 0 && a.lse != nullptr && live) a.lse[(size_t)r * H + hr] = lse;
        } else {
            const size_t ub = (size_t)d.unit;
            // 256 fp32 dims per head: two passes of 128 dims (one 512-byte staged row)
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(c.tmem + kTmemO + lane_base + 128 * hf + 32 * cc, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(stage_addr(c, h, 8 * cc + q), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
                stage_flush(c, warp, lane, [&](int hh) { return (p.pair ? (hh & 63) : hh) < H; },
                            [&](int hh) { return p.po + ((ub * 2 + c.half) * p.lanes + hh) * 256 + 128 * hf; });
            }
            if (hr < H) __stcg(p.ml + (ub * 2 + c.half) * p.lanes + h, make_float2(m_used, lsum));
        }
        // All TMEM reads of O are complete (tcgen05.wait::ld) before the next
        // unit's Q is staged; its first PV (which overwrites O) waits for Q.
        tc_fence_before();
        side0_bar();
    }
    if (!ok) err |= SMLA_DEV_TIMEOUT;
}

// ---------------------------------------------------------------------------
// plan helpers (prologue, all threads of the CTA)
// ---------------------------------------------------------------------------
// The row holding tile position pos of the concatenated stream (the last r
// with cum[r] <= pos; rows with no tile are skipped over by cum).
__device__ __forceinline__ int row_of_tile(const int* cum, int R, long long pos) {
    int lo = 0, hi = R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= pos) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The equal range q (of Q ranges [q T / Q, (q + 1) T / Q)) holding pos, and
// the start of range q; 32-bit division when T * Q fits (64-bit integer
// division is a long software sequence).
__device__ __forceinline__ int stream_range_of(long long pos, long long T, int Q) {
    if (T * Q < (1LL << 32)) return (int)(((uint32_t)(pos + 1) * (uint32_t)Q - 1u) / (uint32_t)T);
    return (int)(((pos + 1) * Q - 1) / T);
}
__device__ __forceinline__ long long stream_range_start(int q, long long T, int Q) {
    if (T * Q < (1LL << 32)) return (long long)(((uint32_t)q * (uint32_t)T) / (uint32_t)Q);
    return (long long)q * T / Q;
}

// The range holding tile position pos (0 <= pos < cut[Q]) of strictly
// increasing cuts cut[0] = 0 < cut[1] < ... < cut[Q]: the last q < Q with
// cut[q] <= pos.
__device__ __forceinline__ int cut_range_of(const int* cut, int Q, long long pos) {
    int lo = 0, hi = Q - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cut[mid] <= pos) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// out[r] = sum of f(r') for r' < r, r < R, and out[R] = the total; one warp,
// lane l takes the contiguous rows [l per, (l + 1) per).
template <class F>
__device__ void warp_exclusive_scan(int R, int* out, F f) {
    const int lane = threadIdx.x & 31;
    const int per = (R + 31) / 32;
    const int r0 = min(R, lane * per), r1 = min(R, r0 + per);
    int my_sum = 0;
    for (int r = r0; r < r1; ++r) my_sum += f(r);
    int incl = my_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - my_sum;
    for (int r = r0; r < r1; ++r) {
        const int v = f(r);  // read before out[r] is written: f may read out
        out[r] = run;
        run += v;
    }
    if (lane == 31) out[R] = incl;
    __syncwarp();
}

// The split plan, on one warp.  Two candidates, chosen by an estimated
// makespan in tiles (each unit also costs about kUnitCostTiles of staging and
// finishing):
//  (a) chunked: tiles_r per row; smallest chunk c with
//      sum_r max(1, ceil(tiles_r / c)) <= budget; row r gets
//      s_r = ceil(tiles_r / ceil(tiles_r / ceil(tiles_r / c))) equal splits and
//      pair p takes units p, p + n_pairs, ...  The budget is the caller's
//      rows * num_splits, rounded down to a whole number of passes over the
//      grid's pairs when it exceeds one pass.
//  (b) stream: the rows' tiles laid end to end and cut into Q equal ranges,
//      one per pair; a row crossing a cut gets one unit per range it meets
//      (at most rows + Q - 1 units, which the workspace always holds).  Rows
//      with no tile get one empty unit each, on pair r % Q.
// Writes this pair's unit list and its length (misc[2]).
__device__ void plan_warp(const KParams& p, int pair, int n_pairs, UnitDesc* units, volatile uint32_t* misc,
                          int* s_tiles, int* s_prefix, int* s_cum, int* s_cut, int* s_eacc, uint32_t& plan_err) {
    const smla_decode_args& a = p.a;
    const int lane = threadIdx.x & 31;
    const int R = p.vrows;  // work rows
    const int budget = max(R, p.units > n_pairs ? (p.units / n_pairs) * n_pairs : p.units);
    int max_t = 1;
    for (int r = lane; r < R; r += 32) {
        const int t = vrow_tiles(make_vrow(p, r, plan_err));
        s_tiles[r] = t;
        max_t = max(max_t, t);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) max_t = max(max_t, __shfl_xor_sync(0xffffffffu, max_t, o));
    __syncwarp();
    warp_exclusive_scan(R, s_cum, [&](int r) { return s_tiles[r]; });
    const long long T = s_cum[R];
    // candidate (b), first: Q ranges, each at least kMinStreamTiles tiles long
    int Q = min(min(n_pairs, p.unit_cap - R + 1), kMaxStreamRanges);
    Q = (int)min((long long)Q, max(1LL, T / kMinStreamTiles));
    bool stream_ok = false;
    long long mk_s = 0;
    if (Q > 1 && T > 0) {
        // Equal cuts first.  A range that meets e more rows than one pays about
        // e * kUnitCostTiles more (staging and finishing its extra units), so
        // the cuts then move to give it that many fewer tiles: cut q sits at
        // q L - kUnitCostTiles * (e_0 + ... + e_{q-1}), L = (T + kUnitCostTiles E) / Q.
        // They are kept only if every range stays non-empty.  e_q counts the
        // rows (with tiles) that start strictly inside range q: one pass over
        // the rows, not a search per range.
        for (int q = lane; q <= Q; q += 32) s_cut[q] = 0;
        __syncwarp();
        for (int r = lane + 1; r < R; r += 32) {
            const long long b0 = s_cum[r];
            if (s_tiles[r] == 0 || b0 >= T) continue;
            const int q = stream_range_of(b0, T, Q);
            if (stream_range_start(q, T, Q) != b0) atomicAdd(&s_cut[q], 1);
        }
        __syncwarp();
        warp_exclusive_scan(Q, s_eacc, [&](int q) { return s_cut[q]; });
        const long long E = s_eacc[Q];
        for (int q = lane; q <= Q; q += 32)
            s_cut[q] = q == Q ? (int)T
                              : (int)(((long long)q * (T + kUnitCostTiles * E) - (long long)kUnitCostTiles * Q * s_eacc[q]) / Q);
        __syncwarp();
        bool inc = true;
        for (int q = lane; q < Q; q += 32) inc = inc && s_cut[q] < s_cut[q + 1];
        if (!__all_sync(0xffffffffu, inc)) {
            for (int q = lane; q <= Q; q += 32) s_cut[q] = (int)stream_range_start(q, T, Q);
        }
        // each range's units on the final cuts (the row holding its first tile
        // plus the rows starting inside it) and the estimated makespan
        for (int q = lane; q <= Q; q += 32) s_eacc[q] = 1;
        __syncwarp();
        for (int r = lane + 1; r < R; r += 32) {
            const int b0 = s_cum[r];
            if (s_tiles[r] == 0 || b0 >= T) continue;
            const int q = cut_range_of(s_cut, Q, b0);
            if (s_cut[q] != b0) atomicAdd(&s_eacc[q], 1);
        }
        __syncwarp();
        int zero_rows = 0, upp = 0;
        for (int r = lane; r < R; r += 32) zero_rows += s_tiles[r] == 0;
        for (int q = lane; q < Q; q += 32) {
            upp = max(upp, s_eacc[q]);
            mk_s = max(mk_s, (long long)(s_cut[q + 1] - s_cut[q]) + (long long)kUnitCostTiles * s_eacc[q]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            zero_rows += __shfl_xor_sync(0xffffffffu, zero_rows, o);
            upp = max(upp, __shfl_xor_sync(0xffffffffu, upp, o));
            mk_s = max(mk_s, __shfl_xor_sync(0xffffffffu, mk_s, o));
        }
        const int zero_share = min(zero_rows, (R + Q - 1) / Q);  // empty rows r = q, q + Q, ... of one pair
        upp += zero_share;
        mk_s += (long long)kUnitCostTiles * zero_share;
        stream_ok = upp <= kMaxUnitsPerPair;
    }
    // Candidate (a) only when it can win.  With a budget of at most one pass
    // over the pairs its makespan is chunk + kUnitCostTiles, and the chunk is at
    // least T / budget (the budget's units must cover every tile); a stream
    // makespan below that bound wins without computing the chunks.
    bool stream = stream_ok && p.units <= n_pairs &&
                  mk_s < (T + budget - 1) / budget + (long long)kUnitCostTiles;
    if (!stream) {
        int lo = 1, hi = max_t;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            long long cnt = 0;
            for (int r = lane; r < R; r += 32) cnt += max(1, ceil_div_i(s_tiles[r], mid));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            if (cnt <= budget) hi = mid; else lo = mid + 1;
        }
        const int chunk = lo;
        warp_exclusive_scan(R, s_prefix, [&](int r) {
            const int t = s_tiles[r];
            int sr = max(1, ceil_div_i(t, chunk));
            if (t > 0) sr = ceil_div_i(t, ceil_div_i(t, sr));
            return sr;
        });
        const int units_c = s_prefix[R];
        const long long passes_c = (units_c + n_pairs - 1) / n_pairs;
        const long long mk_c = (long long)chunk * passes_c + kUnitCostTiles * passes_c;
        // Also over several passes: a chunk count that leaves the last pass
        // part-empty costs the chunked plan up to a whole chunk of imbalance and
        // many partials, which one range per pair avoids.
        stream = stream_ok && mk_s < mk_c;
    }
    if (stream) {
        // per-row unit counts of the stream plan, then (in place) their prefix: unit ids
        for (int r = lane; r < R; r += 32) {
            const int t = s_tiles[r];
            s_prefix[r] = t == 0 ? 1 : cut_range_of(s_cut, Q, s_cum[r + 1] - 1) - cut_range_of(s_cut, Q, s_cum[r]) + 1;
        }
        __syncwarp();
        warp_exclusive_scan(R, s_prefix, [&](int r) { return s_prefix[r]; });
    }
    const int total_units = s_prefix[R];
    if (blockIdx.x == 0)  // the merge kernel's map of the partials
        for (int r = lane; r < R; r += 32) p.row_table[r] = make_int2(s_prefix[r], s_prefix[r + 1] - s_prefix[r]);
    if (lane == 0) {
        int n = 0;
        if (stream) {
            if (pair < Q) {
                const long long ra = s_cut[pair], rb = s_cut[pair + 1];
                if (ra < rb) {
                    for (int r = row_of_tile(s_cum, R, ra); r < R && s_cum[r] < rb; ++r) {
                        if (s_tiles[r] == 0) continue;
                        const int q0 = cut_range_of(s_cut, Q, s_cum[r]);
                        UnitDesc d;
                        d.row = r;
                        d.row_u0 = s_prefix[r];
                        d.s_r = s_prefix[r + 1] - d.row_u0;
                        d.unit = d.row_u0 + (pair - q0);
                        d.t_begin = (int)(max(ra, (long long)s_cum[r]) - s_cum[r]);
                        d.t_end = (int)(min(rb, (long long)s_cum[r + 1]) - s_cum[r]);
                        d.pad0 = d.pad1 = 0;
                        if (n < kMaxUnitsPerPair) units[n++] = d;
                    }
                }
                for (int r = pair; r < R; r += Q) {
                    if (s_tiles[r] != 0) continue;
                    UnitDesc d;
                    d.row = r;
                    d.row_u0 = d.unit = s_prefix[r];
                    d.s_r = 1;
                    d.t_begin = d.t_end = 0;
                    d.pad0 = d.pad1 = 0;
                    if (n < kMaxUnitsPerPair) units[n++] = d;
                }
            }
        } else {
            // this pair's units: pair, pair + n_pairs, ...
            for (int u = pair; u < total_units && n < kMaxUnitsPerPair; u += n_pairs, ++n) {
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
                const int Tr = s_tiles[l2];
                const int tps = Tr > 0 ? ceil_div_i(Tr, d.s_r) : 0;
                d.t_begin = min(Tr, (u - d.row_u0) * tps);
                d.t_end = min(Tr, d.t_begin + tps);
                d.pad0 = d.pad1 = 0;
                units[n] = d;
            }
        }
        misc[2] = (uint32_t)n;
        if (n > 0) {  // the first unit's q rows start their trip to L2 now
            const int rr0 = p.pair ? 2 * units[0].row : units[0].row;
            const int nr = (p.pair && rr0 + 1 < a.num_rows) ? 2 : 1;
            const size_t r0 = (size_t)rr0 * a.num_heads;
            bulk_prefetch_l2(static_cast<const uint16_t*>(a.q_nope) + r0 * SMLA_NOPE_DIMS,
                             (uint32_t)(nr * a.num_heads * SMLA_NOPE_DIMS * 2));
            bulk_prefetch_l2(static_cast<const uint16_t*>(a.q_rope) + r0 * SMLA_ROPE_DIMS,
                             (uint32_t)(nr * a.num_heads * SMLA_ROPE_DIMS * 2));
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) smla_decode_kernel(const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx c;
    c.sb = smem_addr(smem);
    c.half = blockIdx.x & 1u;
    c.wait_ns = p.wait_ns;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc);
    c.abort = misc + 1;
    int* s_tiles = reinterpret_cast<int*>(smem + kOffRaw);  // prologue only
    int* s_prefix = s_tiles + SMLA_MAX_ROWS;                 // [R + 1]
    int* s_cum = s_prefix + SMLA_MAX_ROWS + 1;               // [R + 1]
    int* s_cut = s_cum + SMLA_MAX_ROWS + 1;                  // [Q + 1] stream-plan cuts
    int* s_eacc = s_cut + kMaxStreamRanges + 1;              // [Q + 1]
    UnitDesc* units = reinterpret_cast<UnitDesc*>(smem + kOffUnits);
    const int pair = blockIdx.x >> 1;
    const int n_pairs = gridDim.x >> 1;

    uint32_t err = 0;
    if (tid == 0) {
        misc[1] = 0u;
        for (int i = 0; i < kNR; ++i) {
            mbar_init(bar_addr(c, BAR_RAW_FULL + i), 33);  // 32 async (cp.async) + 1 (producer lane 0)
            mbar_init(bar_addr(c, BAR_RAW_EMPTY + i), kNumDequantWarps);
        }
        for (int i = 0; i < kNXO; ++i) {
            mbar_init(bar_addr(c, BAR_X_FULL + i), kNumDequantWarps);
            mbar_init(bar_addr(c, BAR_XO_EMPTY + i), 1);
        }
        mbar_init(bar_addr(c, BAR_XP_EMPTY), 1);
        mbar_init(bar_addr(c, BAR_XP_FULL), kNumDequantWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_addr(c, BAR_S_FULL + i), 1);
            mbar_init(bar_addr(c, BAR_S_PEER + i), 1);
            mbar_init(bar_addr(c, BAR_S_PEER_READ + i), kSoftmaxWarps);
            mbar_init(bar_addr(c, BAR_P_FULL + i), kSoftmaxWarps);
        }
        mbar_init(bar_addr(c, BAR_O_DONE), 1);
        mbar_init(bar_addr(c, BAR_O_DONE + 1), 1);
        mbar_init(bar_addr(c, BAR_Q_READY), kSideWarps);
        mbar_init(bar_addr(c, BAR_MMA_FINAL), 1);
        // the tensor core's commits and the bulk copies arrive on these
        // barriers through the async proxy: their initialisation is released
        // to it before first use
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(c.sb + kOffMisc, kTmemCols);
        tmem_relinquish();
    }
    // Start every row's q on its way to L2 while the plan runs (pair p takes
    // rows p, p + pairs, ...): the first units' Q staging then reads L2.
    if (warp == kPlanWarp + 1 && lane == 0) {
        const int H = p.a.num_heads;
        for (int r = pair; r < p.a.num_rows; r += n_pairs) {
            bulk_prefetch_l2(static_cast<const uint16_t*>(p.a.q_nope) + (size_t)r * H * SMLA_NOPE_DIMS,
                             (uint32_t)(H * SMLA_NOPE_DIMS * 2));
            bulk_prefetch_l2(static_cast<const uint16_t*>(p.a.q_rope) + (size_t)r * H * SMLA_ROPE_DIMS,
                             (uint32_t)(H * SMLA_ROPE_DIMS * 2));
        }
    }

    // ---- in-kernel split plan (identical in every CTA; reads live lengths),
    //      computed by one warp while the others set up barriers and TMEM ----
    uint32_t plan_err = 0;
    if (warp == kPlanWarp) plan_warp(p, pair, n_pairs, units, misc, s_tiles, s_prefix, s_cum, s_cut, s_eacc, plan_err);
    if (blockIdx.x == 0 && plan_err) err |= plan_err;
    tc_fence_before();
    __syncthreads();  // barrier inits, TMEM address and unit list visible; plan scratch dead
    tc_fence_after();
    c.tmem = misc[0];
    const int n_units = (int)misc[2];

    if (warp < kSoftmaxWarps) {
        softmax_role(p, c, units, n_units, err);
    } else if (warp < kProducerWarp0 + kNumProducers) {
        producer_role(p, c, units, n_units, warp - kProducerWarp0, err);
        if (c.half != 0) err &= ~(SMLA_DEV_BAD_INDEX | SMLA_DEV_BAD_CMP);  // reported once, by half 0
    } else if (warp == kMmaWarp) {
        if (lane == 0) mma_role(c, units, n_units);
        __syncwarp();
    } else {
        dequant_role(c, units, n_units, warp - kDequantWarp0, p.pair != 0);
    }

    tc_fence_before();
    __syncthreads();
    if (*c.abort) err |= SMLA_DEV_TIMEOUT;
    if (err != 0u) atomicOr(p.err, err);
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(c.tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// merge kernel: the partials of split rows -> bf16 out + lse
// ---------------------------------------------------------------------------
// One block per (row, dims half, group of kMergeHeads heads), spread over the
// whole GPU; rows with one partial were finished by the decode kernel and are
// skipped.  Thread = (head, 8 dims): the 32 threads of a head read its 1 KB
// row of each partial.  Each thread merges the partials in split order with a
// running maximum (one pass: every load of a partial is independent of the
// others): with M = max(sink, m_0..m_i) so far, Z and acc are kept scaled to
// 2^-M and rescaled when M grows; at the end out = acc / Z and
// lse = (M + log2 Z) ln 2, equal to the two-pass
// Z = sum_i l_i 2^(m_i - M) + 2^(sink - M), out = sum_i 2^(m_i - M) O_i / Z.
// Partials with m = -inf saw no entry and add nothing (their O is not used);
// a NaN in a used partial reaches the output.
constexpr int kMergeHeads = 8;
constexpr int kMergeThreads = 32 * kMergeHeads;

__global__ void __launch_bounds__(kMergeThreads) smla_merge_kernel(const KParams p) {
    const smla_decode_args& a = p.a;
    const int v = blockIdx.x, half = blockIdx.y, H = a.num_heads, Lw = p.lanes;
    const int lh = blockIdx.z * kMergeHeads + (int)(threadIdx.x >> 5), q = threadIdx.x & 31;  // lane of the work row
    const int2 rt = p.row_table[v];
    const int u0 = rt.x, sr = rt.y;
    const int r = p.pair ? 2 * v + (lh >> 6) : v;  // the row and head this lane holds
    const int h = p.pair ? (lh & 63) : lh;
    if (sr <= 1 || lh >= Lw || h >= H || r >= a.num_rows) return;
    const size_t ml_step = 2 * (size_t)Lw, po_step = 2 * (size_t)Lw * 256;  // one unit
    const float2* ml = p.ml + ((size_t)u0 * 2 + half) * Lw + lh;
    const float* po = p.po + (((size_t)u0 * 2 + half) * Lw + lh) * 256 + 8 * q;
    const float sink2 = a.sink != nullptr ? __ldg(a.sink + h) * kLog2e : -INFINITY;
    float M = sink2, Z = sink2 != -INFINITY ? 1.f : 0.f, lall = 0.f;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 4
    for (int i = 0; i < sr; ++i) {
        // O is loaded beside (m, l), so that the loads of successive partials
        // overlap: every partial slot of the row was written by its unit
        const float2 mi = __ldcg(ml + i * ml_step);
        const float4 x0 = __ldcg(reinterpret_cast<const float4*>(po + i * po_step));
        const float4 x1 = __ldcg(reinterpret_cast<const float4*>(po + i * po_step) + 1);
        lall += mi.y;
        if (mi.x == -INFINITY) continue;  // saw no entry: its O is not used
        if (mi.x > M) {  // the running maximum grows: rescale what is summed so far
            const float f = M == -INFINITY ? 0.f : exp2f(M - mi.x);
            Z *= f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] *= f;
            M = mi.x;
        }
        const float w = exp2f(mi.x - M);
        Z += mi.y * w;
        acc[0] += w * x0.x; acc[1] += w * x0.y; acc[2] += w * x0.z; acc[3] += w * x0.w;
        acc[4] += w * x1.x; acc[5] += w * x1.y; acc[6] += w * x1.z; acc[7] += w * x1.w;
    }
    const float inv = Z > 0.f ? 1.f / Z : 0.f;
    uint4 o;
    o.x = pack_bf16(acc[0] * inv, acc[1] * inv); o.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16(acc[4] * inv, acc[5] * inv); o.w = pack_bf16(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + ((size_t)r * H + h) * SMLA_HEAD_DIM + 256 * half + 8 * q) = o;
    if (half == 0 && q == 0 && a.lse != nullptr) {
        float lse = (M == -INFINITY || Z <= 0.f) ? -INFINITY : (M + log2f(Z)) * kLn2;
        if (lall == 0.f) lse = a.sink != nullptr ? __ldg(a.sink + h) : -INFINITY;  // sink only, exactly
        a.lse[(size_t)r * H + h] = lse;
    }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
namespace {
std::atomic<int> g_attr_done[64];
std::atomic<int> g_resident[64];  // co-resident CTAs of the kernel per device
std::mutex g_attr_mu;

cudaError_t ensure_kernel_attrs(int dev) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_attr_done[dev].load(std::memory_order_acquire) == 1) return cudaSuccess;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (g_attr_done[dev].load(std::memory_order_relaxed) == 1) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(smla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, smla_decode_kernel, kThreads, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_resident[dev].store(std::max(2, per_sm * sms), std::memory_order_relaxed);
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
    kp.row_table = reinterpret_cast<int2*>(ws + L.off_rows);
    kp.ml = reinterpret_cast<float2*>(ws + L.off_ml);
    kp.po = reinterpret_cast<float*>(ws + L.off_po);
    kp.pair = pair_rows(args->num_heads) ? 1 : 0;
    kp.vrows = work_rows(args->num_rows, args->num_heads);
    kp.lanes = partial_lanes(args->num_heads);
    kp.units = kp.vrows * args->num_splits;
    kp.unit_cap = unit_capacity(kp.vrows, args->num_splits);
    kp.wait_ns = wait_limit_ns();
    // Persistent grid: CTA pairs (one CTA per output half) up to what is
    // co-resident (the stream plan can use every one of them), and enough
    // pairs that the chunked plan hands none more than kMaxUnitsPerPair units.
    const int pairs_resident = std::max(1, g_resident[dev].load(std::memory_order_relaxed) / 2);
    int pairs = std::min(kp.unit_cap, pairs_resident);
    pairs = std::max(pairs, (kp.units + kMaxUnitsPerPair - 1) / kMaxUnitsPerPair);
    const dim3 grid((unsigned)(2 * pairs)), block(kThreads);
    smla_decode_kernel<<<grid, block, kSmemBytes, stream>>>(kp);
    if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
    // split rows: a second launch merges their partials across the whole GPU
    const dim3 mgrid((unsigned)kp.vrows, 2u, (unsigned)((kp.lanes + kMergeHeads - 1) / kMergeHeads));
    smla_merge_kernel<<<mgrid, kMergeThreads, 0, stream>>>(kp);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
