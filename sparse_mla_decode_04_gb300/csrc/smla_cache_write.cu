// Cache writer: latent rows (bf16, 448 NoPE + 64 RoPE dims) -> the decode's
// cache layout (448 e4m3 bytes + 64 bf16, one UE8M0 code per 64 NoPE dims).
//
// Method ("[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on gfx950",
// section "Design", last paragraph): the writers cap UE8M0 codes at 254 and
// canonicalise RoPE NaNs.  Per 64-dim group the code is the smallest power of
// two that brings the group's largest magnitude within the e4m3 range (448),
// clamped to [0, 254]; each value is stored as e4m3(x * 2^(127 - code)),
// rounded to nearest, ties to even, saturating at +-448.  A NaN NoPE value is
// stored as 0x7F, a value that rounds to zero as 0x00, a NaN RoPE value as
// the canonical bf16 NaN 0x7FC0; every other RoPE value is copied unchanged.
//
// One warp per row: lane l < 28 converts NoPE dims [16 l, 16 l + 16) (group
// l / 4, its amax reduced over 4 lanes), lanes 28..31 copy 16 RoPE dims each.
// The path is HBM-bound: 1024 bytes read and 584 written per row.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kRowsInFlight = 2;  // rows a warp loads before converting any

// Smallest code c in [0, 254] with amax <= 448 * 2^(c - 127), from the fp32
// bits of amax (>= 0, not NaN): amax = m 2^e, 448 = 1.75 2^8, so
// c = 127 + e - 8 + [m > 1.75], clamped; +inf gives the cap.
__device__ __forceinline__ uint32_t ue8m0_code(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int be = (int)(b >> 23);  // biased exponent
    if (be == 255) return 254u;
    if (be == 0) return 0u;  // zero or subnormal: 448 x 2^-127 already covers it
    const int c = be - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return (uint32_t)min(max(c, 0), 254);
}

// 2^(127 - code) as fp32 (code 254 gives the subnormal 2^-127).
__device__ __forceinline__ float inv_scale(uint32_t code) {
    return code <= 253u ? __uint_as_float((254u - code) << 23) : __uint_as_float(0x00400000u);
}

// Four values -> four e4m3 bytes (lowest byte = a).  The conversion rounds to
// nearest even and saturates finite values at +-448 (0x7E); a NaN comes out
// with magnitude 0x7F and loses its sign here, and a zero of either sign
// becomes 0x00, four bytes at a time: for a magnitude m <= 0x7F, bit 7 of
// m + 0x7F is set iff m != 0 and bit 7 of m + 1 iff m == 0x7F (no carry leaves
// a byte).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    const uint32_t r = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3) |
                       ((uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3) << 16);
    const uint32_t mag = r & 0x7F7F7F7Fu;
    const uint32_t nonzero = (mag + 0x7F7F7F7Fu) & 0x80808080u;
    const uint32_t nan = (mag + 0x01010101u) & 0x80808080u;
    return r & ((nonzero >> 7) * 0xFFu) & ~nan;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Every NaN of two bf16 values becomes 0x7FC0, both halves at once: for a
// magnitude m <= 0x7FFF, bit 15 of m + 0x7F is set iff m > 0x7F80 (a NaN), and
// the low half's sum never carries into the high half.
__device__ __forceinline__ uint32_t canon_nan_bf16x2(uint32_t w) {
    const uint32_t nan = ((w & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u;
    const uint32_t mask = (nan >> 15) * 0xFFFFu;
    return (w & ~mask) | (0x7FC07FC0u & mask);
}

// Two products a * f, b * f in one packed fp32x2 multiply (each lane rounds
// as the scalar multiply does).
__device__ __forceinline__ float2 mul2(float a, float b, float f) {
    uint64_t x, y, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(f));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}

// One row: w holds this lane's 16 dims (dims 16 lane .. 16 lane + 15).
__device__ __forceinline__ void write_row(const uint32_t (&w)[8], int lane, uint8_t* dst, uint8_t* sdst) {
    // every lane takes part in the group reductions (shuffles); RoPE lanes
    // contribute a dummy zero that never leaves their own 4-lane group
    // |x| maxima on bf16 pairs (a NaN is passed over, as fmaxf does)
    __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
    if (lane < 28) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t a = w[i] & 0x7FFF7FFFu;
            __nv_bfloat162 v;
            memcpy(&v, &a, 4);
            m2 = __hmax2(m2, v);
        }
    }
    float amax = fmaxf(__low2float(m2), __high2float(m2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint32_t code = ue8m0_code(amax);
    if (lane < 28) {
        const float f = inv_scale(code);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p0 = mul2(bf16_lo(w[2 * i]), bf16_hi(w[2 * i]), f);
            const float2 p1 = mul2(bf16_lo(w[2 * i + 1]), bf16_hi(w[2 * i + 1]), f);
            o[i] = e4m3x4(p0.x, p0.y, p1.x, p1.y);
        }
        __stcs(reinterpret_cast<uint4*>(dst + 16 * lane), make_uint4(o[0], o[1], o[2], o[3]));
    } else {
        uint4 r0, r1;
        r0.x = canon_nan_bf16x2(w[0]); r0.y = canon_nan_bf16x2(w[1]);
        r0.z = canon_nan_bf16x2(w[2]); r0.w = canon_nan_bf16x2(w[3]);
        r1.x = canon_nan_bf16x2(w[4]); r1.y = canon_nan_bf16x2(w[5]);
        r1.z = canon_nan_bf16x2(w[6]); r1.w = canon_nan_bf16x2(w[7]);
        uint4* rd = reinterpret_cast<uint4*>(dst + SMLA_NOPE_DIMS + 32 * (lane - 28));
        __stcs(rd, r0);
        __stcs(rd + 1, r1);
    }
    // the 7 codes (held by lanes 0, 4, ..., 24) and a zero pad byte, one 8-byte
    // store: group g's first lane places its code at byte g of the pair
    const int g = lane >> 2;
    const bool first = (lane & 3) == 0 && g < 7;
    const uint32_t lo = __reduce_or_sync(0xffffffffu, (first && g < 4) ? code << (8 * g) : 0u);
    const uint32_t hi = __reduce_or_sync(0xffffffffu, (first && g >= 4) ? code << (8 * (g - 4)) : 0u);
    if (lane == 0) *reinterpret_cast<uint2*>(sdst) = make_uint2(lo, hi);
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock) smla_cache_write_kernel(
    const uint4* __restrict__ latent, int64_t num_rows, const int64_t* __restrict__ slots, uint8_t* __restrict__ pool,
    uint8_t* __restrict__ scales, int64_t n_pool, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerBlock;
    uint32_t bad = 0;
    // kRowsInFlight rows per warp step, all their loads issued before any is used
    for (int64_t row0 = warp0; row0 < num_rows; row0 += kRowsInFlight * nwarps) {
        uint32_t w[kRowsInFlight][8];
        int64_t sl[kRowsInFlight];
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u) {
            const int64_t row = row0 + u * nwarps;
            sl[u] = -1;
            if (row < num_rows) {
                sl[u] = __ldcs(slots + row);
                const uint4 v0 = __ldcs(latent + row * 64 + 2 * lane);      // dims 16 l .. 16 l + 7
                const uint4 v1 = __ldcs(latent + row * 64 + 2 * lane + 1);  // dims 16 l + 8 .. 16 l + 15
                w[u][0] = v0.x; w[u][1] = v0.y; w[u][2] = v0.z; w[u][3] = v0.w;
                w[u][4] = v1.x; w[u][5] = v1.y; w[u][6] = v1.z; w[u][7] = v1.w;
            }
        }
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u) {
            const int64_t s = sl[u];  // -1 also for rows past the end
            if (s == -1) continue;    // warp-uniform
            if (s < -1 || s >= n_pool) {
                bad = 1;
                continue;
            }
            write_row(w[u], lane, pool + s * SMLA_ENTRY_BYTES, scales + s * SMLA_SCALE_BYTES);
        }
    }
    if (err != nullptr && __any_sync(0xffffffffu, bad != 0) && lane == 0) atomicOr(err, SMLA_DEV_BAD_INDEX);
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace smla

extern "C" smla_status smla_cache_write(const void* latent, int64_t num_rows, const int64_t* slots, void* pool,
                                        void* scales, int64_t n_pool, uint32_t* dev_error, smla_stream_t stream) {
    using namespace smla;
    if (num_rows < 0 || n_pool < 0) return SMLA_ERR_BAD_SHAPE;
    if (num_rows == 0) return SMLA_OK;
    if (latent == nullptr || slots == nullptr || pool == nullptr || scales == nullptr) return SMLA_ERR_NULL_POINTER;
    if (!aligned_to(latent, 16) || !aligned_to(pool, 16) || !aligned_to(slots, 8) || !aligned_to(scales, 8) ||
        !aligned_to(dev_error, 4))
        return SMLA_ERR_MISALIGNED;
    const smla_status dev = check_device_only();
    if (dev != SMLA_OK) return dev;
    int sms = 0, d = 0, per_sm = 0;
    if (cudaGetDevice(&d) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, smla_cache_write_kernel, 32 * kWarpsPerBlock, 0) !=
            cudaSuccess)
        return SMLA_ERR_CUDA;
    // one resident wave of blocks, each warp striding over the rows
    const int64_t blocks_needed = (num_rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int blocks = (int)std::min<int64_t>(blocks_needed, (int64_t)sms * std::max(1, per_sm));
    smla_cache_write_kernel<<<blocks, 32 * kWarpsPerBlock, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(latent), num_rows, slots, static_cast<uint8_t*>(pool), static_cast<uint8_t*>(scales),
        n_pool, dev_error);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}
