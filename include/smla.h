/*
 * smla.h — C ABI of the GB300 (sm_103a) sparse multi-head latent attention
 * (MLA) decode library, libsmla.so.
 *
 * What is computed (one decode step).  Each query row r has H heads that
 * share one latent KV pool.  Row r attends to a multiset of entries, in this
 * order: the valid slots of its top-k index list into the main cache, its
 * sliding window, and its compressed-cache entries.  Each entry holds 448
 * FP8-e4m3 NoPE dims with one UE8M0 scale per 64 dims and 64 bf16 RoPE dims;
 * dequantised, it is a 512-wide vector x_e used as both key and value.  For
 * head h with query q_h = [q_nope | q_rope] (512 wide):
 *
 *     s_e   = sm_scale * <q_h, x_e>
 *     lse_h = ln( e^{sink_h} + sum_e e^{s_e} )        (natural log, sink included)
 *     out_h = sum_e e^{s_e - lse_h} * x_e             (512 wide, bf16)
 *
 * Sources: "[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on gfx950"
 * (vLLM pull request 52212), section "Design": the 512-wide combined
 * NoPE + RoPE QK dot, the 512-wide PV, guarded main/window tiles, compressed
 * 64-entry groups with masked tails, attention sinks, invalid indices with
 * zero probability, 64-bit block address arithmetic; and "[ASM] [HIP] [MLA v4
 * nm] Split plan helper and persistent decode kernel with in-kernel split and
 * merge" (ROCm/aiter pull request 6126), summary part 1 (host split planner
 * from a cost model) and part 2 (split plan computed in the kernel from the
 * real lengths on every call; split rows merged from fp32 partials plus LSE;
 * unsplit rows write bf16 directly; CUDA-graph safe with varying lengths; the
 * workspace is allocated outside capture and calls sharing it are
 * stream-ordered).  There the last-arriving work-group of a row merges it
 * inside the one launch; here a second launch merges every split row at once
 * across the whole GPU, which keeps the merge off the decode kernel's tail.
 *
 * Threading: every function is thread-safe.  The library allocates no device
 * memory and keeps no per-call state; the caller owns every buffer.
 */
#ifndef SMLA_H_
#define SMLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (a cudaStream_t / CUstream); NULL = legacy default stream. */
typedef void* smla_stream_t;

typedef enum smla_status {
    SMLA_OK = 0,
    SMLA_ERR_NULL_POINTER = 1,        /* a required pointer is NULL                    */
    SMLA_ERR_MISALIGNED = 2,          /* a pointer breaks its stated alignment          */
    SMLA_ERR_BAD_SHAPE = 3,           /* rows / heads / topk / splits / sizes out of range */
    SMLA_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes < smla_workspace_bytes(...)           */
    SMLA_ERR_UNSUPPORTED_DEVICE = 5,  /* current device is not compute capability 10.3  */
    SMLA_ERR_CUDA = 6                 /* a CUDA runtime call or the launch failed       */
} smla_status;

/* Bits of the device error word (smla_read_device_error).  Bad device data
 * never traps: the offending slot is treated as invalid (zero probability)
 * and a bit is set. */
#define SMLA_DEV_BAD_INDEX   0x1u  /* top-k index < -1, or a logical position that does not map into the pool */
#define SMLA_DEV_BAD_CMP     0x2u  /* compressed range outside [0, n_cmp): the excess is dropped */
#define SMLA_DEV_BAD_LENGTH  0x4u  /* negative swa_len / cmp_len: treated as 0 */
#define SMLA_DEV_TIMEOUT     0x8u  /* a bounded wait inside the kernel gave up; outputs of the
                                      call are undefined */

/* Fixed geometry of one KV entry. */
#define SMLA_NOPE_DIMS   448
#define SMLA_ROPE_DIMS   64
#define SMLA_HEAD_DIM    512  /* QK width and PV width */
#define SMLA_ENTRY_BYTES 576  /* 448 fp8 bytes followed by 64 little-endian bf16 */
#define SMLA_SCALE_BYTES 8    /* 7 UE8M0 codes (one per 64 NoPE dims) + 1 pad byte */
#define SMLA_PAGE_SIZE   64   /* tokens per page of block_table */
#define SMLA_MAX_HEADS   128
#define SMLA_MAX_ROWS    1024
#define SMLA_MAX_SPLITS  32

/*
 * Arguments of one decode call.  All pointers are DEVICE pointers owned by
 * the caller.  Layouts are C-contiguous.  bf16 arrays are given as raw 16-bit
 * storage.  Required alignments: q_nope, q_rope, kv_pool, cmp_pool, out 16 B;
 * kv_scales, cmp_scales 8 B; every int32 / float array 4 B.
 */
typedef struct smla_decode_args {
    const void* q_nope;          /* bf16 [num_rows][num_heads][448]                                */
    const void* q_rope;          /* bf16 [num_rows][num_heads][64]                                 */
    const void* kv_pool;         /* u8   [n_main][576]: main-cache entries                          */
    const void* kv_scales;       /* u8   [n_main][8]:   UE8M0 codes, scale = 2^(code-127)           */
    int64_t n_main;              /* rows in kv_pool (may exceed 2^31 / 576: addressing is 64-bit)   */
    const int32_t* block_table;  /* [num_seqs][pages_per_seq] physical page ids, or NULL: logical
                                    position == physical row.  Position p of sequence s lives in
                                    row block_table[s][p/64]*64 + p%64.                             */
    int32_t pages_per_seq;       /* row stride of block_table (ignored when it is NULL)             */
    const int32_t* row_seq;      /* [num_rows] sequence of each row, or NULL: row r reads sequence r */
    const int32_t* main_idx;     /* [num_rows][topk] logical positions, -1 = invalid slot           */
    int32_t topk;                /* 0 disables the top-k source (main_idx may then be NULL)          */
    const int32_t* swa_start;    /* [num_rows] first logical position of the sliding window          */
    const int32_t* swa_len;      /* [num_rows] window length; NULL disables the window              */
    const void* cmp_pool;        /* u8 [n_cmp][576]: compressed-cache entries                        */
    const void* cmp_scales;      /* u8 [n_cmp][8]                                                    */
    int64_t n_cmp;               /* rows in cmp_pool                                                 */
    const int32_t* cmp_start;    /* [num_rows] first compressed row of the row                       */
    const int32_t* cmp_len;      /* [num_rows] compressed entries of the row; NULL disables them     */
    const float* sink;           /* [num_heads] per-head sink logit (scaled domain), NULL = no sink  */
    float sm_scale;              /* softmax scale applied to <q, x>                                  */
    void* out;                   /* bf16 [num_rows][num_heads][512]                                  */
    float* lse;                  /* [num_rows][num_heads] natural-log LSE incl. sink, or NULL        */
    int32_t num_rows;            /* 1 .. SMLA_MAX_ROWS                                               */
    int32_t num_heads;           /* 1 .. SMLA_MAX_HEADS                                              */
    int32_t num_splits;          /* 1 .. SMLA_MAX_SPLITS: split budget per row (from the planner).
                                    The kernel's chunked plan uses at most num_rows*num_splits work
                                    units, handed to rows in proportion to each row's live length;
                                    its stream plan instead cuts the rows' tiles, laid end to end,
                                    into one equal range per CTA pair (a row crossing a cut is
                                    merged from its parts).  The kernel takes whichever plan has the
                                    smaller estimated time, from the live lengths.  Keep num_splits
                                    fixed across CUDA-graph replays.                                 */
} smla_decode_args;

/*
 * Host-side split planner.  Cost model (aiter pull request 6126, summary
 * part 1): choose s in [1, SMLA_MAX_SPLITS] minimising
 *     waves(num_rows * s) * (t0 + c_entry * ceil(kv_len / s))
 *       + [s > 1] * (c_byte * num_rows * num_heads * 512 * 4 * s + c_merge),
 * waves(u) = ceil(u / slots); ties go to the smaller s.  kv_len is the
 * caller's per-row entry count (top-k slots + window + compressed entries).
 * Pure host code: no device work, no allocation.  Returns s >= 1, or the
 * negated smla_status (SMLA_ERR_BAD_SHAPE) for num_rows < 1, num_heads not in
 * [1, 128] or kv_len < 0.
 */
int smla_plan_num_splits(int num_rows, int num_heads, int64_t kv_len);

/* The planner's coefficients; the built-in set is fitted for GB300. */
typedef struct smla_plan_coeffs {
    double slots;    /* work units that run concurrently (one unit = one CTA pair) */
    double t0;       /* fixed time per unit, microseconds                           */
    double c_entry;  /* time per KV entry per unit, microseconds                    */
    double c_byte;   /* partial write + read-back cost, microseconds per byte       */
    double c_merge;  /* fixed merge cost of a split call, microseconds              */
} smla_plan_coeffs;

/* Copies the built-in GB300 coefficients into *out.  Returns SMLA_OK or SMLA_ERR_NULL_POINTER. */
smla_status smla_plan_default_coeffs(smla_plan_coeffs* out);

/* Same cost model with caller-supplied coefficients (NULL = built-in) and an
 * upper bound s_max in [1, SMLA_MAX_SPLITS].  Same return convention. */
int smla_plan_num_splits_ex(int num_rows, int num_heads, int64_t kv_len,
                            const smla_plan_coeffs* coeffs, int s_max);

/*
 * Workspace bytes for calls with up to max_rows rows, num_heads heads and a
 * split budget of max_splits (cf. the persistent kernel's workspace getter in
 * aiter pull request 6126, summary part 2).  The layout is: a device error
 * word, a per-row table of partials (rewritten by every call), per-unit fp32
 * partial (m, l) and per-unit fp32 partial O, for
 * max(max_rows * max_splits, max_rows + 95) units (the second term lets the
 * stream plan use up to 96 CTA pairs).  Allocate it once and zero it once
 * (cudaMemset 0, for the error word), outside any graph capture; it carries
 * no other state between calls, so it can be reused across calls and batch
 * sizes.  Returns 0 for arguments out of range.
 */
size_t smla_workspace_bytes(int max_rows, int num_heads, int max_splits);

/*
 * One decode step: validates on the host, then enqueues two kernel launches
 * on `stream`: the decode kernel, a persistent grid of CTA pairs (one CTA per
 * output dim half, as many as are co-resident on the device), which writes
 * unsplit rows' out and lse and split rows' fp32 partials; then the merge
 * kernel, one block per (row, dim half, 8 heads), which combines the partials
 * of split rows.
 * Host checks come first: NULL or misaligned pointers, unsupported sizes, a
 * workspace smaller than smla_workspace_bytes(num_rows, num_heads, num_splits)
 * and a device that is not sm_103 each return an error and launch nothing.
 * Device-side lengths and indices may change between CUDA-graph replays; bad
 * device data sets bits in the workspace error word (SMLA_DEV_*) and never
 * traps.  Rows with no valid entry get out = 0 and lse = sink (written).
 * Calls that share a workspace must be ordered on one stream.
 * Returns SMLA_OK once both launches are enqueued.
 */
smla_status smla_decode(const smla_decode_args* args, void* workspace, size_t ws_bytes,
                        smla_stream_t stream);

/*
 * Copies the workspace's device error word to *flags (host) and clears it.
 * Enqueued on `stream` and synchronised with it before returning.
 */
smla_status smla_read_device_error(void* workspace, uint32_t* flags, smla_stream_t stream);

/*
 * Diagnostic: sets the limit of every wait inside the decode kernel (each
 * pipeline stage waits for the previous one with a bounded wait) for the
 * launches that follow, in nanoseconds; 0 restores the default of 2 s.
 * Returns the previous limit.  When a wait runs out, the kernel stops all its
 * roles, lets the work it already issued finish, sets SMLA_DEV_TIMEOUT in the
 * workspace error word and returns; the outputs of that call are undefined,
 * and the next call (with a working limit) is unaffected.  Process-wide;
 * thread-safe.  Meant for tests of that path: with the default limit a wait
 * runs out only if the GPU stops making progress.
 */
uint64_t smla_set_wait_limit_ns(uint64_t ns);

/* Static, NUL-terminated description of a status code. */
const char* smla_status_string(smla_status status);

/*
 * Cache writer: quantises latent rows into the cache layout smla_decode reads.
 * Source: "[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on gfx950"
 * (vLLM pull request 52212), section "Design", last paragraph: the cache
 * writers store FP8 NoPE with UE8M0 scales, cap the codes at 254 and
 * canonicalise RoPE NaNs.  For each row i with slots[i] >= 0:
 *   - NoPE group g (dims 64g .. 64g+63, g < 7): code_g = the smallest c in
 *     [0, 254] with max|x| <= 448 * 2^(c-127) (254 when none fits);
 *     pool[s][d] = e4m3(x[d] * 2^(127-code_g)), round to nearest even,
 *     saturating at +-448; a NaN value -> 0x7F; a value rounding to zero -> 0x00;
 *     scales[s][g] = code_g, scales[s][7] = 0;
 *   - RoPE: pool[s][448 + 2i .. ] = x[448 + i] (bf16, little-endian), a NaN
 *     becoming 0x7FC0.
 * Arguments (DEVICE pointers, caller-owned): latent bf16 [num_rows][512]
 * (16-byte aligned); slots int64 [num_rows] (8-byte aligned), -1 = skip the
 * row; pool u8 [n_pool][576] (16-byte aligned) and scales u8 [n_pool][8]
 * (8-byte aligned), written in place; dev_error: optional uint32 word (NULL
 * or 4-byte aligned) that gets SMLA_DEV_BAD_INDEX for a slot < -1 or >= n_pool
 * (that row is skipped).  Two rows with the same slot race.  Host checks as
 * for smla_decode; num_rows = 0 launches nothing.  One kernel launch on
 * `stream`; allocates nothing.
 */
smla_status smla_cache_write(const void* latent, int64_t num_rows, const int64_t* slots, void* pool,
                             void* scales, int64_t n_pool, uint32_t* dev_error, smla_stream_t stream);

/* Largest k accepted by smla_topk_indices. */
#define SMLA_TOPK_MAX_K 4096

/*
 * Top-k producer: the decode's top-k index list from per-position scores.
 * The vLLM page names this step (the indexer top-k path whose cp-gather its
 * comment "8k/1k TP8 follow-up", item 2, reworks) but not how its
 * scores are made, so the scores are an input.  For each row r:
 * out[r][0 .. k-1] = the positions p in [0, min(lens[r], stride)) with the
 * largest scores[r][p], ordered by score descending and then by position
 * ascending (-0 equals +0); positions with a NaN score are never taken; slots
 * left over when fewer than k positions are selectable hold -1.
 * Arguments (DEVICE pointers, caller-owned, 4-byte aligned): scores float32
 * [num_rows][stride]; lens int32 [num_rows]; out int32 [num_rows][k].
 * 1 <= k <= SMLA_TOPK_MAX_K, 0 <= stride < 2^31.  One kernel launch on
 * `stream` (a cluster of two CTAs per row, each over half of it); allocates
 * nothing.
 */
smla_status smla_topk_indices(const float* scores, int64_t stride, const int32_t* lens, int32_t num_rows,
                              int32_t k, int32_t* out, smla_stream_t stream);

/* Bytes of the scratch array built into the library for smla_decode_static_scratch
 * (48 MiB).  It holds the workspace layout of smla_workspace_bytes: with
 * U = max(num_rows * num_splits, num_rows + 95) partial units of
 * num_heads * 2064 bytes each, plus 8.5 KB.  At 128 heads that is U <= 190:
 * num_rows <= 95 and num_rows * num_splits <= 190 (the 32-row x 128-head
 * DeepSeek-V4-like decode fits at up to 5 splits). */
#define SMLA_STATIC_SCRATCH_BYTES (48u * 1024u * 1024u)

/*
 * smla_decode for callers that cannot allocate device memory.  The cited
 * pull-request pages have no counterpart to this entry point.
 *
 * Some callers have no way to call cudaMalloc: plugin or custom-op interfaces
 * that hand a kernel only its inputs, outputs and a stream; code that runs
 * while a CUDA graph is being captured (cudaMalloc is not a stream operation);
 * processes whose device memory is owned entirely by another allocator.  This
 * entry point allocates nothing: its scratch (the same layout as the
 * smla_decode workspace) is a file-scope __device__ array of
 * SMLA_STATIC_SCRATCH_BYTES (48 MiB) that every GPU which loads the library
 * holds until the process exits.  The caller still passes every input and
 * output in `args`.
 *
 * - Calls whose smla_workspace_bytes(num_rows, num_heads, num_splits) exceeds
 *   SMLA_STATIC_SCRATCH_BYTES return SMLA_ERR_WORKSPACE_TOO_SMALL and launch
 *   nothing.  The workspace always holds at least num_rows + 95 units, so
 *   lowering num_splits helps only while num_rows * num_splits is the larger
 *   term; beyond the limit given with SMLA_STATIC_SCRATCH_BYTES, split the
 *   batch into several calls.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture on the device.
 * - Every call on a device shares the one array, and the array keeps what the
 *   last call left.  Each call clears the error word (and the row table) on
 *   `stream` before its launch, so the SMLA_DEV_* flags of a call cannot be
 *   read back through this entry point.  Calls that overlap on the GPU (other
 *   streams, other host threads) race on the array: order them on one stream.
 * - Every host check of smla_decode runs first, before the array is looked up
 *   or written; it returns the same status smla_decode would (after the size
 *   check above).  Otherwise it behaves as smla_decode.
 */
smla_status smla_decode_static_scratch(const smla_decode_args* args, smla_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* SMLA_H_ */
