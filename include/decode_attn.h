/*
 * decode_attn.h - C ABI of the paged grouped-query decode attention library
 * (libpaged_gqa_decode.so, CUDA kernels for sm_103a).
 *
 * The operation (one decode step, one query token per sequence):
 *   for every batch entry b and query head hq, with KV head h = hq / G,
 *   G = Hq / Hkv, L = seq_lens[b] and lo = (window > 0) ? max(0, L - window) : 0,
 *     out[b][hq][:] = sum_{t in [lo, L)} softmax_t(scale * q[b][hq] . k_t) * v_t
 *   where k_t = k_pages[page_table[b][t / PS]][t % PS][h][:] (likewise v_t).
 * Defined by: apache/tvm pull request 20426 "webgpu-decode-attention"
 * (sharded-nest commit: paged decode attention, shards of the context with
 * online-softmax states merged afterwards, short contexts in one pass, the
 * nest chosen on the host; PR description: sliding windows), and
 * BackendStack21/mlx-runner pull request 3, commit "GQA-shared split
 * attention" (one K/V row read serves every query head of its GQA group;
 * split partials merged in a fixed order by a combine kernel).
 *
 * Layouts (all row-major, contiguous, device memory unless stated; "fp16"
 * reads bf16 when params.dtype is DECODE_ATTN_DTYPE_BF16):
 *   q           [B][Hq][D]              fp16   ([B][T][Hq][D] with num_queries T > 1)
 *   k_pages     [P][PS][Hkv][D]         fp16   (the caller's paged cache)
 *   v_pages     [P][PS][Hkv][D]         fp16
 *   page_table  [B][max_pages_per_seq]  int32  (physical page of each logical page)
 *   seq_lens    [B]                     int32  (positions to attend, the new
 *                                                token's K/V already in the cache)
 *   out         [B][Hq][D]              fp16   ([B][T][Hq][D] with num_queries T > 1)
 * Ownership: the caller owns every buffer, including the workspace; the
 * library allocates no device memory and keeps no per-call state (only a
 * per-device cache of the SM count).  Entry points are thread-safe.
 * Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 * default stream); nothing synchronises the host.
 * Device: every call runs on the calling thread's current CUDA device
 * (cudaGetDevice); the pointers and the stream must belong to it.
 * Errors: a negative return means nothing was launched (bad argument) or a
 * CUDA runtime error was reported while launching; decode_attn_strerror()
 * names it.  Problems only the device can see (a page id outside [0, P) in
 * an attended range, a length outside [0, max_pages_per_seq * PS] or above
 * max_seq_len) are OR-ed as DECODE_ATTN_DEV_* bits into *err_flag (when
 * err_flag is not NULL) and the affected output rows are written as zeros;
 * the kernels never trap.
 */
#ifndef PAGED_GQA_DECODE_ATTN_H
#define PAGED_GQA_DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define DECODE_ATTN_OK 0
#define DECODE_ATTN_ERR_NULL (-1)       /* a required pointer is NULL */
#define DECODE_ATTN_ERR_SHAPE (-2)      /* non-positive size, Hq % Hkv != 0, ... */
#define DECODE_ATTN_ERR_HEAD_DIM (-3)   /* head_dim not in {64, 128, 256} */
#define DECODE_ATTN_ERR_PAGE_SIZE (-4)  /* page_size not a power of two in [8, 256] */
#define DECODE_ATTN_ERR_GROUP (-5)      /* G = Hq / Hkv above 16 */
#define DECODE_ATTN_ERR_WORKSPACE (-6)  /* workspace missing or smaller than required */
#define DECODE_ATTN_ERR_ALIGN (-7)      /* a tensor pointer is not 16-byte aligned */
#define DECODE_ATTN_ERR_CUDA (-8)       /* CUDA runtime error (device query or launch) */
#define DECODE_ATTN_ERR_TENSOR_MAP (-9) /* the TMA descriptor for the K/V pool was rejected */
#define DECODE_ATTN_ERR_VARIANT (-10)   /* requested kernel variant cannot run this shape */

/* Device error bits OR-ed into *err_flag. */
#define DECODE_ATTN_DEV_BAD_LEN 1       /* seq_len < 0 or > max_pages_per_seq * page_size */
#define DECODE_ATTN_DEV_BAD_PAGE 2      /* page id outside [0, num_pages) in an attended range */
#define DECODE_ATTN_DEV_OVER_HINT 4     /* seq_len beyond the max_seq_len the grid was planned for */
#define DECODE_ATTN_DEV_TIMEOUT 8       /* a bounded wait gave up (a pipeline wait after about
                                           2 s, a cluster exchange after about 4 s); row zeroed */
#define DECODE_ATTN_DEV_CHECK 32        /* checked build only (libpaged_gqa_decode_checked.so):
                                           an index fell outside its buffer; that access was
                                           skipped (or pointed at the zero-fill coordinate) */
#define DECODE_ATTN_DEV_WORKSPACE 16    /* a group's shard ticket was not zero on entry:
                                           the group's rows may be stale; clear and retry */

/* Element formats of q, k_pages, v_pages, out, k_new, v_new (params.dtype). */
#define DECODE_ATTN_DTYPE_FP16 0        /* IEEE binary16 */
#define DECODE_ATTN_DTYPE_BF16 1        /* bfloat16 (tensor-core variant) */

/* Work schedules of the split kernel (decode_attn_params.schedule). */
#define DECODE_ATTN_SCHEDULE_AUTO 0       /* planner picks (grid, or cluster where it gains) */
#define DECODE_ATTN_SCHEDULE_GRID 1       /* one CTA per (shard, KV head, sequence); the
                                             last CTA of a group merges via the workspace */
#define DECODE_ATTN_SCHEDULE_CLUSTER 2    /* grid schedule whose shards of one (KV head,
                                             sequence) form a thread-block cluster and merge
                                             through distributed shared memory; one-wave
                                             split plans of 2..16 shards, tensor-core variant */

/* Kernel variants (decode_attn_params.variant). */
#define DECODE_ATTN_VARIANT_AUTO 0      /* planner picks */
#define DECODE_ATTN_VARIANT_SIMT 1      /* CUDA-core q.k / p.v with warp-shuffle reductions */
#define DECODE_ATTN_VARIANT_MMA 2       /* tensor-core mma.sync q.k / p.v */

typedef struct decode_attn_params {
  int32_t batch;             /* B >= 0 */
  int32_t num_q_heads;       /* Hq > 0 */
  int32_t num_kv_heads;      /* Hkv > 0, Hq % Hkv == 0, G = Hq / Hkv <= 16 */
  int32_t head_dim;          /* D in {64, 128, 256} */
  int32_t page_size;         /* PS: power of two in [8, 256] */
  int32_t max_pages_per_seq; /* columns of page_table (> 0) */
  int32_t num_pages;         /* P: pages in k_pages / v_pages (> 0) */
  int32_t max_seq_len;       /* host-known bound on seq_lens, sizes the grid;
                                <= 0 means max_pages_per_seq * page_size */
  float scale;               /* multiplies q . k before the softmax */
  int32_t window;            /* <= 0: whole context; else the last min(L, window) positions */
  int32_t variant;           /* DECODE_ATTN_VARIANT_*; 0 = automatic */
  int32_t split_min;         /* contexts above this use shards + combine; <= 0 means 256;
                                a context longer than one shard holds (1024 boxes of
                                min(page_size, 64) positions) is split regardless */
  int32_t force_chunk;       /* > 0: tokens per shard (rounded up to 64); 0 = planner */
  int32_t num_queries;       /* T new query positions per sequence (<= 0 means 1); with
                                T > 1, q and out are [B][T][Hq][D], query t of sequence b
                                sits at position seq_lens[b] - T + t and attends causally
                                (up to itself; the window counted from it); needs
                                T * G <= 16 and the tensor-core variant */
  int32_t dtype;             /* DECODE_ATTN_DTYPE_*: element format of every 16-bit
                                tensor; accumulation is fp32 for both */
  int32_t schedule;          /* DECODE_ATTN_SCHEDULE_*; 0 = automatic */
} decode_attn_params;

/* Launch plan chosen by the host heuristic (exposed for inspection/tests). */
typedef struct decode_attn_plan {
  int32_t split;             /* 0: single pass writes out; 1: shards + combine */
  int32_t variant;           /* DECODE_ATTN_VARIANT_SIMT or _MMA */
  int32_t group_pad;         /* G rounded up to the kernel's head group (1,2,4,8,16) */
  int32_t tile_tokens;       /* tokens per pipeline stage (64) */
  int32_t chunk_tokens;      /* C: tokens per shard, a multiple of tile_tokens */
  int32_t max_shards;        /* S_max: shards of the longest planned sequence */
  int32_t grid_x, grid_y, grid_z;  /* split-kernel grid: (kv head, shard, batch) when
                                      head_fastest, else (shard, kv head, batch) */
  int32_t ctas_per_sm;       /* resident CTAs per SM the grid was sized for */
  int32_t head_fastest;      /* grid schedule order: 1 for plans of several waves */
  int32_t ring_stages;       /* 64-token K/V stages in flight per CTA: 3 (6 at D=64);
                                2 (4 at D=64) for grids of several waves of short
                                shards, which fit 3 CTAs per SM (tensor-core variant) */
  int32_t cluster;           /* CTAs per thread-block cluster (the shards of one
                                (KV head, sequence), merged through distributed shared
                                memory; 2..16), or 0 (merged through the workspace) */
  int32_t balanced;          /* 1: each sequence's attended range is cut into max_shards
                                near-equal shards of whole 64-position tiles (chunk_tokens
                                is then an upper bound); 0: shards of chunk_tokens
                                positions (one-wave split plans take 1) */
  size_t workspace_bytes;    /* tickets max(64 KiB, (B*Hkv+64)*4) + partials B*Hq*S_max*(D+2)*4,
                                each part rounded up to 256 B; 0 for a single-pass plan */
} decode_attn_plan;

/*
 * Host heuristic (apache/tvm pull request 20426: the nest is picked on the
 * host, sharded above 256 tokens; BackendStack21/mlx-runner pull request 3:
 * split at context >= a threshold, 256 by default).  Reads only *p and
 * num_sms; touches no device.  Returns DECODE_ATTN_OK or a negative code.
 */
int decode_attn_make_plan(const decode_attn_params* p, int32_t num_sms, decode_attn_plan* plan);

/* Workspace bytes decode_attn needs for *p on `device` (queries its SM
 * count once).  Returns 0 for a single-pass plan or an invalid *p. */
size_t decode_attn_workspace_size(const decode_attn_params* p, int device);

/*
 * One decode step: the host plan, then one split-kernel launch on `stream`.
 * A split plan writes each shard's online-softmax partial to the workspace;
 * the last CTA of each (sequence, KV head) group to finish (an atomic ticket,
 * nothing waits) merges that group's partials in ascending shard order and
 * writes out.  A single-pass plan writes out directly.
 * workspace: device memory of at least decode_attn_workspace_size() bytes,
 * 256-byte aligned, owned by the caller.  Its first 64 KiB (more for plans
 * with over 16384 (sequence, KV head) groups) hold one shard ticket per
 * group, which must be zero when a split launch starts: zero the workspace
 * when allocating it, or call decode_attn_workspace_clear().  Every
 * completed call leaves the tickets zero again, and partials never use that
 * region, so one zeroed buffer serves calls of any shape; after a call that
 * reported DECODE_ATTN_DEV_TIMEOUT or DECODE_ATTN_DEV_WORKSPACE, clear it
 * before reuse.  The rest of the workspace is scratch.  Calls sharing a
 * workspace must not overlap on the GPU.
 * err_flag: nullable device int32, bits DECODE_ATTN_DEV_* are OR-ed in (the
 * caller clears it).  All tensor pointers must be 16-byte aligned.
 */
int decode_attn(const decode_attn_params* p, const void* q, const void* k_pages,
                const void* v_pages, const int32_t* page_table, const int32_t* seq_lens,
                void* out, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                void* stream);

/*
 * decode_attn_split: the kernel launch decode_attn makes (same arguments,
 * same result; kept as its own entry point so the split kernel can be timed
 * or captured alone).  decode_attn_combine: re-merges the partials that the
 * last split launch with this workspace left behind into out, in ascending
 * shard order, as a separate kernel launched as a programmatic dependent of
 * the preceding kernel on the stream; it runs the same merge code as the
 * split kernel's last CTAs and gives the same bits.  A no-op returning
 * DECODE_ATTN_OK for a single-pass plan.  The plan is recomputed from *p and
 * must match the split call's.
 */
int decode_attn_split(const decode_attn_params* p, const void* q, const void* k_pages,
                      const void* v_pages, const int32_t* page_table, const int32_t* seq_lens,
                      void* out, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                      void* stream);
int decode_attn_combine(const decode_attn_params* p, const int32_t* seq_lens, void* out,
                        void* workspace, size_t workspace_bytes, int32_t* err_flag,
                        void* stream);

/*
 * Paged K/V append, the step before attention (idle-intelligence/llm-web
 * pull request 8, suffix-prefill commit: the new K/V rows are scattered into
 * the cache at their positions after the resident prefix).  For every b with
 * positions[b] >= 0 and every KV head h:
 *   k_pages[page_table[b][t / PS]][t % PS][h][:] = k_new[b][h][:],  t = positions[b]
 * (likewise v).  k_new, v_new: [B][Hkv][D] fp16 device; positions: [B] int32
 * device.  Uses batch, num_kv_heads, head_dim, page_size, max_pages_per_seq
 * and num_pages of *p (the other fields must still be valid).  Bit-exact copy.
 * A position past the table raises DECODE_ATTN_DEV_BAD_LEN, a page id
 * outside [0, P) DECODE_ATTN_DEV_BAD_PAGE; that sequence is not written.
 */
int decode_kv_append(const decode_attn_params* p, const void* k_new, const void* v_new,
                     const int32_t* positions, void* k_pages, void* v_pages,
                     const int32_t* page_table, int32_t* err_flag, void* stream);

/*
 * Append + attention in one launch: the same result as decode_kv_append with
 * positions[b] = seq_lens[b] - 1 (the new token is the last attended
 * position; sequences with seq_len 0 get no row) followed by decode_attn.
 * The CTA holding each sequence's last position writes the new rows of its
 * KV head before it streams its tiles.  Arguments as decode_attn plus k_new,
 * v_new ([B][Hkv][D] fp16 device); k_pages and v_pages are written.
 */
int decode_attn_append(const decode_attn_params* p, const void* q, const void* k_new,
                       const void* v_new, void* k_pages, void* v_pages,
                       const int32_t* page_table, const int32_t* seq_lens, void* out,
                       void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream);

/*
 * End-to-end step from HOST buffers: enqueues the host-to-device copies of
 * q, k_pages, v_pages, page_table and seq_lens into the caller's device
 * buffers (d_* arguments, same layouts), decode_attn, and the device-to-host
 * copy of out into out_host.  Host buffers should be pinned for the copies to
 * be asynchronous.  Nothing synchronises: the caller waits on `stream`
 * before reading out_host.  kv_bytes_to_copy: bytes of each of k_pages and
 * v_pages to copy (the pool prefix in use); 0 copies the whole pool.
 */
int decode_attn_host(const decode_attn_params* p, const void* q_host, const void* k_pages_host,
                     const void* v_pages_host, const int32_t* page_table_host,
                     const int32_t* seq_lens_host, void* out_host, void* d_q, void* d_k_pages,
                     void* d_v_pages, int32_t* d_page_table, int32_t* d_seq_lens, void* d_out,
                     size_t kv_bytes_to_copy, void* workspace, size_t workspace_bytes,
                     int32_t* err_flag, void* stream);

/* Zeroes the shard tickets of a workspace sized for *p (an async memset on
 * `stream`); DECODE_ATTN_OK without work for a single-pass plan. */
int decode_attn_workspace_clear(const decode_attn_params* p, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Static text for a return code. */
const char* decode_attn_strerror(int status);

/*
 * ---- Variant that allocates nothing (the pages have no counterpart) ----
 *
 * decode_attn_static_scratch: the same step as decode_attn, for callers that
 * cannot allocate device memory themselves (their device memory is held by
 * another framework's allocator, they sit behind a plugin interface that
 * passes only the call's tensors, or they must not pay cudaMalloc's implicit
 * synchronisation).  The shard partials go to a fixed array of
 * DECODE_ATTN_STATIC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.  The caller still passes
 * the inputs and the output (layouts, alignment and err_flag as for
 * decode_attn).  The first call on a device looks up the array's device
 * address on that device; make that first call before any stream capture.
 * Plans whose partials need more than the array return
 * DECODE_ATTN_ERR_SCRATCH_LIMIT without launching; decode_attn_workspace_size
 * tells the need in advance.  All calls on a device share the array: calls
 * whose GPU work can overlap (other streams, other host threads) race and
 * must be serialised by the caller.  The array keeps the last call's
 * contents; the only part that must start at zero, the shard tickets, is
 * cleared by each call itself (an asynchronous memset on `stream` before the
 * launch), so nothing needs clearing by the caller, also after a call that
 * reported DECODE_ATTN_DEV_TIMEOUT.  Calls no cudaMalloc, cudaFree or
 * allocating routine.
 */
#define DECODE_ATTN_STATIC_SCRATCH_BYTES (8u << 20)
#define DECODE_ATTN_ERR_SCRATCH_LIMIT (-11) /* partials above the static scratch size */
int decode_attn_static_scratch(const decode_attn_params* p, const void* q, const void* k_pages,
                               const void* v_pages, const int32_t* page_table,
                               const int32_t* seq_lens, void* out, int32_t* err_flag,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_GQA_DECODE_ATTN_H */
