/*
 * mla_verify.h -- C ABI of the DDTree verify-attention library (MLA, absorbed
 * form) for GB300 / sm_103a.
 *
 * The operation.  Speculative decoding with a draft tree verifies all Q tree
 * nodes of a sequence in one attention call.  Each (node i, head h) query row
 * attends over the whole committed prefix plus the tree nodes that are node i
 * itself or its ancestors ("Ground Truth in Silicon: The Role of the Python
 * Reference in Custom CUDA Kernel Development", section "Input Knowledge
 * Required to Understand This Message", item 3; "Reading the Reference: How a
 * Single File-Read Message Anchored a Complex CUDA Kernel Implementation",
 * section "Output Knowledge Created by This Message": prefix visibility plus
 * tree-tail visibility).  The attention is DeepSeek-V3 / Kimi multi-head
 * latent attention in absorbed form: the KV cache holds, per token, a latent
 * kv_c of width 512 and a rope key k_pe of width 64, both shared by every
 * head ("Ground Truth in Silicon ...", section "The Message in Full"; ibid.
 * item 2).  For row (b, i, h) over visible tokens j:
 *
 *     s_j = scale * (q_lat[b,i,h,:] . kv_c[j,:] + q_pe[b,i,h,:] . k_pe[j,:])
 *     lse[b,i,h]   = ln sum_j exp(s_j)
 *     out[b,i,h,:] = sum_j exp(s_j - lse) * kv_c[j,:]            (width 512)
 *
 * The softmax runs online with fp32 accumulation over a bf16 (or fp32) cache
 * ("Reading the Reference ...", section "Why This File Matters": bf16 KV
 * cache, streaming online softmax, prefix and tail masked in one pass).
 *
 * Token placement.  Logical positions of sequence b are 0 .. N_b-1 with
 * N_b = prefix_lens[b] + Q: the prefix first, then tree node t at position
 * prefix_lens[b] + t.  A position maps to a pool slot through either
 *   page_size == 1 : slot = kv_indices[kv_indptr[b] + pos]  (scattered slots,
 *                    as in "The Critical Glue: Validating a Custom Flash
 *                    Attention Kernel Through Test Infrastructure", section
 *                    "The Context"), or
 *   page_size  > 1 : slot = block_table[b][pos / page_size] * page_size
 *                           + pos % page_size.
 *
 * Conventions for every entry point below.
 *   - Pointers inside mla_verify_args, the workspace, and the anc / slots
 *     outputs are DEVICE pointers owned by the caller.  The library keeps no
 *     pointer after a call returns and allocates no memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and never synchronise the host, except mla_verify_check, whose
 *     whole purpose is to read the device error word.
 *   - Argument errors found on the host return before anything is launched.
 *     Errors in device-resident tables (a slot outside the pool, a parent
 *     outside [-1, i-1], an indptr that disagrees with prefix_lens, a page
 *     entry outside the pool) are caught by the metadata kernel, which sets a
 *     bit in the workspace error word; the attention kernels then skip all
 *     work, so no access ever leaves the pool.  mla_verify_check reports them.
 *   - A failed CUDA launch returns MLA_ERR_CUDA.
 */
#ifndef MLA_VERIFY_H
#define MLA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_VERIFY_ABI_VERSION 1
#define MLA_DL 512 /* latent width, fixed */
#define MLA_DR 64  /* rope width, fixed */
#define MLA_MAX_Q 64 /* tree nodes per sequence: one 64-bit ancestor mask */

typedef struct CUstream_st *mla_stream_t; /* same type as cudaStream_t */

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* a host-visible argument is malformed */
    MLA_ERR_UNSUPPORTED = 2,  /* well formed but outside what the kernels do (Q > 64, ...) */
    MLA_ERR_CUDA = 3,         /* a CUDA call or launch failed */
    MLA_ERR_WORKSPACE = 4,    /* workspace NULL, misaligned or smaller than required */
    MLA_ERR_DEVICE_CHECK = 5  /* the device found bad table contents (see mla_verify_check) */
} mla_status;

typedef enum { MLA_BF16 = 0, MLA_FP32 = 1 } mla_dtype;

/* Which kernel family runs the attention.  AUTO takes the tensor-core kernel
 * for bf16 and the CUDA-core kernel for fp32 (fp32 needs fp32 products to meet
 * a 1e-4 relative tolerance).  SIMT forces the CUDA-core kernel for either
 * dtype; TC requires bf16. */
typedef enum { MLA_ALGO_AUTO = 0, MLA_ALGO_SIMT = 1, MLA_ALGO_TC = 2 } mla_algo;

typedef struct {
    int B;                      /* sequences, >= 0 */
    int Q;                      /* draft-tree nodes per sequence, 0..64 (0 = no-op) */
    int H;                      /* heads, >= 1 */
    mla_dtype dtype;            /* element type of q_lat, q_pe, kv_c, k_pe and out */
    const void *q_lat;          /* [B][Q][H][512], contiguous */
    const void *q_pe;           /* [B][Q][H][64], contiguous */
    const void *kv_c;           /* pool row r at element offset r * kv_c_stride (512 used) */
    const void *k_pe;           /* pool row r at element offset r * k_pe_stride (64 used) */
    int64_t kv_c_stride;        /* elements; >= 512, row bytes a multiple of 16 */
    int64_t k_pe_stride;        /* elements; >= 64,  row bytes a multiple of 16 */
    int64_t pool_slots;         /* rows in the pool; every resolved slot must be below it */
    int page_size;              /* 1: kv_indptr/kv_indices;  > 1: block_table */
    const int32_t *kv_indptr;   /* [B+1]; kv_indptr[0] == 0, kv_indptr[b+1]-kv_indptr[b] == prefix_lens[b]+Q */
    const int32_t *kv_indices;  /* [kv_indptr[B]] pool slots */
    const int32_t *block_table; /* [B][max_pages] page ids */
    int max_pages;              /* columns of block_table */
    const int32_t *prefix_lens; /* [B], >= 0 */
    const int32_t *tree_parent; /* [B][Q], parent[i] in [-1, i-1]; -1 hangs off the prefix */
    float scale;                /* score scale, finite and > 0, e.g. 1/sqrt(192) */
    void *out;                  /* [B][Q][H][512] of dtype */
    float *lse;                 /* [B][Q][H], natural log; may be NULL */
    mla_algo algo;              /* kernel family, see mla_algo */
    void *const *profile_events;/* optional, normally NULL: two cudaEvent_t the call records
                                   on `stream` right before and right after the attention
                                   kernel, so a caller can time that kernel alone */
} mla_verify_args;

/* Bytes of device workspace mla_verify_attn needs for these arguments and
 * this num_splits (same meaning as in mla_verify_attn).  Returns 0 when the
 * arguments are invalid or, for num_splits == 0, when no CUDA device can be
 * queried.  Depends only on B, Q, H, dtype, algo and the device's SM count,
 * never on device-resident table contents. */
size_t mla_verify_workspace_size(const mla_verify_args *args, int num_splits);

/* The verify attention.  Enqueues the metadata kernel (tree masks, tile
 * counts, table validation), the split-KV attention kernel, and, where a row
 * group's KV was cut into several pieces, the LSE-combine kernel, all on
 * `stream`.  workspace: device memory of at least
 * mla_verify_workspace_size(args, num_splits) bytes, 256-byte aligned, not
 * used concurrently by another call.  num_splits: n > 0 cuts the KV range
 * of every row group (256 query rows for the tensor-core kernel, 16 for the
 * SIMT kernel) into exactly n chunks, merged by the LSE-combine kernel when
 * n > 1 (a chunk is empty when a sequence has fewer than n KV tiles).  0: the
 * library chooses.  From B, H, Q and the SM count it takes S_max, the count
 * whose work items fill the GPU in whole waves, and sizes the workspace for
 * it; the SIMT kernel uses S_max, while for the tensor-core kernel the
 * metadata kernel, once it has read prefix_lens, picks the count in
 * [1, S_max] that a cost model of the kernels (time per tile and per work
 * item, the combine's pass over the partials) rates fastest -- so the count
 * follows the sequences' lengths without a host synchronisation, and equal
 * inputs always get the same count (read it back with
 * mla_verify_splits_used).  Results do not depend on the split count beyond
 * fp32 rounding. */
mla_status mla_verify_attn(const mla_verify_args *args, void *workspace, size_t ws_bytes,
                           int num_splits, mla_stream_t stream);

/* Same computation as mla_verify_attn, for callers that cannot allocate device
 * memory when they make the call (a plugin inside an engine that owns the
 * whole device memory pool, a decode loop that must not take the device-wide
 * synchronisation of cudaMalloc) and so have no workspace to pass.  The pages
 * have no counterpart of this entry point.
 * It allocates nothing: its workspace is a fixed array of
 * MLA_NOALLOC_SCRATCH_BYTES compiled into the library.  The array is reserved
 * on a device when the library's device code is loaded there, which under
 * lazy module loading (the CUDA default) happens during the first call on that
 * device: make that first call at start-up, before an engine claims the rest
 * of the device memory and before any stream capture.  It stays reserved until
 * the process exits.  Arguments and outputs mean what they mean for
 * mla_verify_attn.  num_splits > 0: that many KV chunks per row group; a call
 * whose mla_verify_workspace_size exceeds MLA_NOALLOC_SCRATCH_BYTES returns
 * MLA_ERR_WORKSPACE before launching anything.  num_splits == 0: the automatic
 * split count, lowered until the workspace fits the array (one split always
 * fits), so the results can differ in fp32 rounding from mla_verify_attn's
 * automatic choice on large problems.  The device address of the array is
 * looked up once per CUDA context (a context created after cudaDeviceReset is
 * looked up again).  All calls share the array and it keeps the previous
 * call's contents (the error word is cleared at the start of each call); calls
 * that overlap on the GPU race on it, so order them on one stream.  Device-side
 * table errors are reported in the array's error word: read it with
 * mla_verify_noalloc_check. */
#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
mla_status mla_verify_attn_noalloc(const mla_verify_args *args, int num_splits, mla_stream_t stream);

/* mla_verify_check for mla_verify_attn_noalloc: synchronises `stream`, then
 * reads the error word the last no-allocation call on the current device left
 * in the library's scratch array.  Returns MLA_OK or MLA_ERR_DEVICE_CHECK (or
 * MLA_ERR_CUDA); *bits (may be NULL) receives the raw MLA_DEVERR_* bits.
 * Allocates nothing.  No counterpart on the pages. */
mla_status mla_verify_noalloc_check(mla_stream_t stream, uint32_t *bits);

/* Parity / debug export of the index work the attention kernels rely on.
 * Runs the metadata kernel and writes
 *   anc   [B][Q] uint64: bit t set when node t is node i or an ancestor of it;
 *   slots [sum_b (prefix_lens[b]+Q)] int32: pool slot of every logical
 *         position, sequences back to back in order;
 * slots_capacity bounds the slots array (entries); positions beyond it are
 * not written and MLA_ERR_INVALID_ARG is recorded in the error word.
 * workspace as for mla_verify_attn with num_splits = 1. */
mla_status mla_verify_build_meta(const mla_verify_args *args, void *workspace, size_t ws_bytes,
                                 uint64_t *anc, int32_t *slots, int64_t slots_capacity,
                                 mla_stream_t stream);

/* Synchronises `stream`, then reads the workspace error word left by the last
 * call that used this workspace.  Returns MLA_OK or MLA_ERR_DEVICE_CHECK (or
 * MLA_ERR_CUDA); *bits (may be NULL) receives the raw MLA_DEVERR_* bits. */
mla_status mla_verify_check(const void *workspace, mla_stream_t stream, uint32_t *bits);

/* Synchronises `stream`, then reads the split count (KV chunks per row group)
 * that the last mla_verify_attn call on this workspace used: num_splits when
 * that was > 0, else the one the library chose (a call with B or Q zero
 * launches nothing and leaves the value unchanged).  Returns
 * MLA_ERR_WORKSPACE for a NULL workspace and MLA_ERR_INVALID_ARG for a NULL
 * `splits`, before touching the device.  Debug and benchmark aid; no
 * counterpart on the pages. */
mla_status mla_verify_splits_used(const void *workspace, mla_stream_t stream, int32_t *splits);

/* KV compaction ("Ground Truth in Silicon ...", section "Why This Message Was
 * Written": KV-cache defragmentation).  For every sequence b and logical
 * position p in [0, prefix_lens[b] + Q) -- prefix first, then the tree nodes,
 * the order mla_verify_attn reads them -- copies the kv_c and k_pe rows of the
 * slot that position resolves to (page_size 1 or paged, as in args) to slot
 * dst_slot0 + base[b] + p of the destination arrays, where base[b] is the sum
 * of the earlier sequences' lengths; writes new_kv_indices[base[b] + p] = that
 * slot and, when new_kv_indptr is not NULL, new_kv_indptr[b] = base[b]
 * (B + 1 entries).  With those two tables and page_size = 1 the verify call on
 * the destination gives the same bytes as on the source.
 *   dst_kv_c, dst_k_pe: device arrays of dst_slots rows, row strides in
 *     elements (>= 512 / >= 64, multiples of 16 bytes), 16-byte aligned, the
 *     cache's dtype; they must not overlap any source row;
 *   dst_slot0 >= 0; dst_slots <= INT32_MAX; rows that would land at or beyond
 *     dst_slots are skipped and MLA_DEVERR_CAPACITY is recorded;
 *   workspace as for mla_verify_attn with num_splits = 1; args as for
 *   mla_verify_attn (queries, outputs and scale are not read).
 * Device-side table errors are reported as for mla_verify_attn
 * (mla_verify_check) and then nothing is copied.  Asynchronous on `stream`. */
mla_status mla_kv_compact(const mla_verify_args *args, void *workspace, size_t ws_bytes, void *dst_kv_c,
                          void *dst_k_pe, int64_t dst_kv_c_stride, int64_t dst_k_pe_stride, int64_t dst_slot0,
                          int64_t dst_slots, int32_t *new_kv_indices, int32_t *new_kv_indptr,
                          mla_stream_t stream);

/* Failure-detection self-test.  Runs mla_verify_attn's tensor-core path
 * (bf16 caches; args->algo AUTO or TC; num_splits automatic) with one extra
 * device wait, at the start of the score MMA role, on a barrier that nothing
 * completes, bounded by hold_ns (0 < hold_ns <= 1e9).  That wait gives up,
 * every CTA of its cluster stops issuing work, drains what it issued and
 * frees its Tensor Memory, and the call completes with MLA_DEVERR_TIMEOUT in
 * the workspace error word (and the wait site in the second 32-bit word);
 * out and lse are not written.  The context stays usable: the next call on
 * the same workspace runs normally.  Returns MLA_ERR_INVALID_ARG for a zero or
 * larger hold_ns or an empty problem, MLA_ERR_UNSUPPORTED for other dtypes or
 * algorithms, otherwise as mla_verify_attn. */
mla_status mla_verify_selftest_timeout(const mla_verify_args *args, void *workspace, size_t ws_bytes,
                                       uint64_t hold_ns, mla_stream_t stream);

#define MLA_DEVERR_PREFIX 0x1u   /* prefix_lens[b] < 0 */
#define MLA_DEVERR_INDPTR 0x2u   /* kv_indptr[0] != 0, or a span != prefix_lens[b] + Q */
#define MLA_DEVERR_SLOT 0x4u     /* resolved slot outside [0, pool_slots) */
#define MLA_DEVERR_PARENT 0x8u   /* tree_parent[b][i] outside [-1, i-1] */
#define MLA_DEVERR_PAGES 0x10u   /* sequence longer than max_pages * page_size */
#define MLA_DEVERR_CAPACITY 0x20u/* build_meta: slots_capacity too small */
#define MLA_DEVERR_TIMEOUT 0x40u /* a bounded device wait gave up */
#define MLA_DEVERR_LAYOUT 0x80u  /* the tensor-core kernel's shared memory was not 1024-byte aligned */

/* Human-readable name of a status code (static storage). */
const char *mla_status_str(mla_status s);

/* MLA_VERIFY_ABI_VERSION of the built library. */
int mla_verify_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_VERIFY_H */
