// Internal declarations shared by the host code and the kernel launcher.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include "smla.h"

namespace smla {

// Workspace layout.  The error word and the row table sit at fixed offsets,
// so that a workspace stays valid across calls with different row counts.
struct WorkspaceLayout {
    size_t off_err;       // uint32 device error word
    size_t off_rows;      // int2 [SMLA_MAX_ROWS] per row: first unit, partials (written by each call)
    size_t off_ml;        // float2 [units][2][H]  per-unit (m, l), one copy per dim half
    size_t off_po;        // float  [units][2][H][256] per-unit unnormalised O by dims half (units = unit_capacity)
    size_t total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Partial slots: rows * splits for the chunked plan, and at least
// rows + kWorkspacePairs - 1 so that the stream plan (one tile range per CTA
// pair, up to kWorkspacePairs pairs) always fits.
constexpr int kWorkspacePairs = 96;
inline int unit_capacity(int rows, int splits) {
    const int a = rows * splits, b = rows + kWorkspacePairs - 1;
    return a > b ? a : b;
}

// With num_heads <= 64 the decode pairs rows 2v and 2v + 1 into one work row
// of 128 TMEM lanes (row A's heads on lanes 0..63, row B's on 64..127); its
// partials then hold 128 lanes.
inline bool pair_rows(int heads) { return heads <= 64; }
inline int work_rows(int rows, int heads) { return pair_rows(heads) ? (rows + 1) / 2 : rows; }
inline int partial_lanes(int heads) { return pair_rows(heads) ? 128 : heads; }

inline WorkspaceLayout workspace_layout(int rows, int heads, int splits) {
    WorkspaceLayout L;
    const size_t units = (size_t)unit_capacity(work_rows(rows, heads), splits);
    heads = partial_lanes(heads);
    L.off_err = 0;
    L.off_rows = 256;
    L.off_ml = align_up(L.off_rows + sizeof(int32_t) * 2 * SMLA_MAX_ROWS, 256);
    L.off_po = align_up(L.off_ml + units * 2 * (size_t)heads * 2 * sizeof(float), 256);
    L.total = L.off_po + units * (size_t)heads * SMLA_HEAD_DIM * sizeof(float);
    return L;
}

// Host checks of smla_decode (defined in smla_host.cpp).  check_decode_args
// covers the argument struct (sizes, NULL and misaligned pointers);
// check_decode_call adds the workspace (NULL, 256-byte alignment, size) and
// the device (compute capability 10.3).  Both return the status smla_decode
// would return, and touch nothing on the device.
smla_status check_decode_args(const smla_decode_args* a);
smla_status check_decode_call(const smla_decode_args* a, const void* workspace, size_t ws_bytes);
// The device check alone (compute capability 10.3, cached per device).
smla_status check_device_only();

// Limit of every pipeline wait inside the decode kernel, in ns (set by
// smla_set_wait_limit_ns; 2 s by default).
uint64_t wait_limit_ns();

// Host-validated launch of the decode and merge kernels (defined in smla_decode.cu).
smla_status launch_decode(const smla_decode_args* args, void* workspace, cudaStream_t stream);

}  // namespace smla
