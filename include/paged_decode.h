/*
 * paged_decode.h -- C ABI of the GB300 (sm_103a) paged decode attention
 * library (libpaged_decode.so).
 *
 * What it computes (FlashInfer "flashinfer.cake_fmha" API page: the paged
 * decode contract trtllm_batch_decode_with_kv_cache(query, kv_cache,
 * workspace_buffer, block_tables, seq_lens, max_kv_len); PR #4557 "Blackwell
 * TRT-LLM MLA decode backend": the MLA call with bmm scales, lse/return_lse,
 * cum_seq_lens_q and max_q_len):
 *
 *   for every request b, query row i < q_len_b, query head h:
 *     g   = h / (Hq / Hkv)                       (MLA: Hkv = 1, g = 0)
 *     pos = seq_lens[b] - q_len_b + i            (keys 0..pos are visible;
 *                                                 PR #4557 review "Exclusive
 *                                                 causal bound drops the
 *                                                 newest key")
 *     key/value row of token t: page block_tables[b][t / P], slot t % P
 *     s_t = sm_scale * k_scale * <q, k_t>;  p = softmax(s)
 *     out[row][h] = v_scale * sum_t p_t v_t ;  lse[row][h] = log sum_t exp(s_t)
 *
 * seq_lens is the total cached length INCLUDING the q_len_b new tokens
 * (PR #5952 commit #5956 "Contract": seq_lens = total length after the
 * append), so q_len_b <= seq_lens[b] is required. LSE is a natural log.
 *
 * Layouts (the pages name NHD and HND; PR #5952 gives NHD's shape):
 *   NHD  pool [num_pages][page_size][Hkv][D]
 *   HND  pool [num_pages][Hkv][page_size][D]
 *   MLA  pool [num_pages][page_size][576]: key = the whole row (512 latent +
 *        64 rope channels, PR #5552), value = its first 512 channels.
 * FP8 storage (PR #5956 "Contract"): K/V hold x / k_scale, x / v_scale as
 * OCP E4M3FN bytes; k_scale and v_scale are fp32 scalars in device memory.
 *
 * Ownership and conventions
 *  - Every device pointer is owned by the caller. The library allocates no
 *    device memory after it is loaded; split partials, work lists and
 *    counters live in a caller-owned workspace whose size the plan reports
 *    (PR #5591: caller-owned workspace, counters that reset themselves).
 *  - A plan is built on the host from host copies of seq_lens / q_indptr. It
 *    keeps no hidden cache keyed on addresses (PR #4557: host metadata must
 *    not outlive the tensors it describes). paged_decode_plan_upload writes
 *    the plan into a workspace; a run then checks on the device that the
 *    workspace holds that plan and that the device seq_lens / q_indptr equal
 *    the plan's, and flags any difference instead of reading stale data.
 *  - Run calls do not synchronise the host and enqueue kernels only (no
 *    copies, no memsets), so they can be captured in a CUDA graph after an
 *    upload done outside the capture.
 *  - Host-detectable errors are returned as pd_status and nothing is
 *    launched. Device-detectable errors (a page id outside [0, num_pages),
 *    metadata that differs from the plan) set an error word in the
 *    workspace, which paged_decode_read_error returns; the rows of an
 *    affected request are written as zeros and no out-of-range address is
 *    read. No kernel traps, and every device wait is bounded.
 *  - No function throws; all are thread-safe for distinct plans.
 */
#ifndef PAGED_DECODE_H
#define PAGED_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers; NULL = legacy stream. */
typedef struct CUstream_st* pd_stream_t;

typedef enum {
  PD_OK = 0,
  PD_ERR_INVALID_ARG = 1,         /* a host argument is out of range          */
  PD_ERR_WORKSPACE_TOO_SMALL = 2, /* workspace_bytes < the plan's requirement */
  PD_ERR_UNSUPPORTED = 3,         /* valid, but a shape this build lacks      */
  PD_ERR_CUDA = 4,                /* a CUDA runtime call failed               */
  PD_ERR_DEVICE_FLAG = 5,         /* read_error: the device flagged an error  */
} pd_status;

typedef enum { PD_LAYOUT_NHD = 0, PD_LAYOUT_HND = 1 } pd_layout;
typedef enum { PD_KV_BF16 = 0, PD_KV_FP8_E4M3 = 1 } pd_kv_dtype;
/* PD_ATTN_PREFILL: GQA attention of many new tokens per request (the
 * pages' context call), run by paged_prefill_run on the tensor cores. */
typedef enum { PD_ATTN_GQA = 0, PD_ATTN_MLA = 1, PD_ATTN_PREFILL = 2 } pd_attn_kind;
/* How split partial states are merged (PR #4557 split-KV reducer; PR #5591
 * last-arriver split merge). */
typedef enum {
  PD_MERGE_AUTO = 0,     /* the library's choice: KERNEL (measured on
                            GB300 no slower than FUSED for GQA decode and
                            faster with many splits; MLA states are 64 rows
                            x 512 channels)                                 */
  PD_MERGE_FUSED = 1,    /* the CTA whose split arrives last merges the unit
                            inside the decode kernel (one launch per call;
                            prefill plans use KERNEL whatever is asked)     */
  PD_MERGE_KERNEL = 2,   /* a separate LSE-merge kernel, launched as a
                            programmatic dependent of the decode kernel     */
} pd_merge_mode;

/* How work items reach the persistent CTAs. */
typedef enum {
  PD_SCHED_AUTO = 0,     /* the planner's choice by predicted finish time        */
  PD_SCHED_STATIC = 1,   /* one equal contiguous range of the (unit, tile)
                            sequence per CTA, cut at unit boundaries           */
  PD_SCHED_QUEUE = 2,    /* equal splits on a shared atomic queue, longest
                            first (PR #4557's persistent CLC work order)       */
} pd_schedule;

/* Device error codes written to the workspace error word. */
typedef enum {
  PD_DEV_OK = 0,
  PD_DEV_BAD_PAGE = 1,       /* a block-table entry outside [0, num_pages)   */
  PD_DEV_SEQ_LEN_MISMATCH = 2, /* device seq_lens[b] differs from the plan  */
  PD_DEV_Q_INDPTR_MISMATCH = 3,/* device q_indptr differs from the plan     */
  PD_DEV_PLAN_MISMATCH = 4,  /* the workspace holds another plan            */
  PD_DEV_TIMEOUT = 5,        /* a bounded device wait gave up               */
} pd_device_error;

/* Problem description. Sizes are element counts unless stated. */
typedef struct {
  int32_t kind;              /* pd_attn_kind                                  */
  int32_t batch;             /* B >= 0 (B = 0 is a no-op)                     */
  int32_t num_q_heads;       /* Hq; MLA: any value >= 1 (128 in DeepSeek-V3)  */
  int32_t num_kv_heads;      /* Hkv, Hq % Hkv == 0; MLA: must be 1            */
  int32_t head_dim_qk;       /* GQA: 128; MLA: 576                            */
  int32_t head_dim_v;        /* GQA: 128 (== head_dim_qk); MLA: 512           */
  int32_t page_size;         /* P >= 1 tokens per page (MLA: a multiple of 8) */
  int32_t num_pages;         /* pool pages; valid page ids are [0, num_pages) */
  int32_t max_pages_per_seq; /* row length of block_tables                    */
  int32_t max_kv_len;        /* upper bound on seq_lens (plan sizing)          */
  int32_t layout;            /* pd_layout (GQA; ignored for MLA)              */
  int32_t kv_dtype;          /* pd_kv_dtype (MLA E4M3: mla_decode_run_fp8)     */
  int32_t max_splits;        /* 1..16 caps the KV splits per unit; 0 = 16     */
  int32_t num_sms;           /* 0 = query the current device                  */
  int32_t merge_mode;        /* pd_merge_mode                                 */
  int32_t schedule;          /* pd_schedule                                   */
  int64_t k_page_stride;     /* elements from page p to p+1 in the K pool;
                                0 = compact (P * Hkv * D, MLA: P * 576)       */
  int64_t v_page_stride;     /* same for the V pool (GQA)                     */
} pd_problem;

typedef struct pd_plan pd_plan;   /* opaque; free with paged_decode_plan_destroy */

/* Summary of a plan (for tests and tooling). */
typedef struct {
  int32_t num_units;       /* independent (request, kv head / row block) units */
  int32_t num_items;       /* work items in the persistent queue              */
  int32_t num_ctas;        /* persistent CTAs launched                        */
  int32_t tile_tokens;     /* tokens per pipeline tile                        */
  int32_t max_splits_used; /* largest number of splits of any unit            */
  int32_t rows_per_unit;   /* query rows a unit carries (<= the kernel's M)   */
  int64_t partial_rows;    /* split partial rows in the workspace             */
  int64_t workspace_bytes; /* size the caller must provide                    */
  uint64_t plan_id;        /* content hash checked on the device              */
  int32_t merge_mode;      /* the pd_merge_mode the plan runs (AUTO resolved) */
  int32_t launches_per_run; /* kernels one run call enqueues: 1, or 2 with the
                               LSE-merge kernel after a split plan           */
} pd_plan_info;

/*
 * Build a plan on the host (no CUDA call other than a device-attribute query
 * when problem->num_sms == 0).
 *   seq_lens_host [batch]   total lengths incl. new tokens; q_len_b <= L_b <=
 *                           max_kv_len <= max_pages_per_seq * page_size
 *   q_indptr_host [batch+1] query rows of request b are
 *                           q_indptr[b] .. q_indptr[b+1]-1; NULL means one
 *                           row per request
 * On success *plan_out owns the plan. Errors: PD_ERR_INVALID_ARG for
 * inconsistent sizes, PD_ERR_UNSUPPORTED for shapes this build lacks.
 * The split planner splits a unit's KV range into at most max_splits
 * contiguous tile ranges (the pages' host never asks for more than 16) and
 * orders the work items longest first (PR #4557 persistent CLC route).
 */
pd_status paged_decode_plan(const pd_problem* problem, const int32_t* seq_lens_host,
                            const int32_t* q_indptr_host, pd_plan** plan_out);

/* Workspace bytes the plan needs (0 for a NULL plan). */
size_t paged_decode_workspace_size(const pd_plan* plan);

pd_status paged_decode_plan_get_info(const pd_plan* plan, pd_plan_info* info);

/* Copy the plan's work items as int32 quadruples (unit, first tile,
 * end tile, split index), in queue order, into items_out[4 * num_items]. */
pd_status paged_decode_plan_get_items(const pd_plan* plan, int32_t* items_out);

/*
 * Write the plan (work list, unit table, zeroed counters and error word)
 * into the workspace with one host-to-device copy on `stream`. Needed once
 * per plan and workspace; runs reuse it. The source is pageable host memory,
 * so do this outside CUDA-graph capture.
 */
pd_status paged_decode_plan_upload(const pd_plan* plan, void* workspace,
                                   size_t workspace_bytes, pd_stream_t stream);

/*
 * GQA / MHA / MQA decode (problem->kind == PD_ATTN_GQA).
 *   q            bf16 [total_q][Hq][D]            (total_q = q_indptr[batch])
 *   k_pool       bf16 or e4m3 pool in the plan's layout, page stride
 *                k_page_stride; 16-byte aligned
 *   v_pool       same layout and element type; may alias a second half of
 *                one combined tensor
 *   block_tables int32 [batch][max_pages_per_seq]; entries past
 *                ceil(L_b / P) are never read
 *   seq_lens     int32 [batch] device copy; must equal the plan's
 *   q_indptr     int32 [batch+1] device copy or NULL (one row per request)
 *   sm_scale     softmax scale applied to q.k
 *   k_scale, v_scale  fp32 device scalars (E4M3 pools) or NULL (bf16 pools)
 *                E4M3 pools are multiplied on f16 tensor cores: each work
 *                item scales its bf16 query rows by one power of two (their
 *                largest magnitude lands in [2^14, 2^15)) before rounding
 *                them to f16, and folds the inverse into the logit scale, so
 *                no finite query saturates; elements more than 2^29 below
 *                the item's largest lose precision in f16
 *   out          bf16 [total_q][Hq][D]
 *   lse          fp32 [total_q][Hq] natural-log LSE, or NULL
 *   workspace    the workspace the plan was uploaded into
 * Enqueues the decode kernel and, when the plan splits a unit and merges
 * with PD_MERGE_KERNEL, the LSE-merge kernel, on `stream`; no host sync.
 */
pd_status paged_decode_run(const pd_plan* plan, const void* q, const void* k_pool,
                           const void* v_pool, const int32_t* block_tables,
                           const int32_t* seq_lens, const int32_t* q_indptr, float sm_scale,
                           const float* k_scale, const float* v_scale, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, pd_stream_t stream);

/*
 * paged_decode_run with attention sinks: sinks is a device fp32
 * [num_q_heads] array of per-head logits (natural-log units, the scale of
 * sm_scale * k_scale * <q, k>) that join the softmax denominator with no
 * value, as the `sinks` argument of the pages' MLA call (PR #4557 review,
 * `_core.py` excerpt; "page64 sink" benchmark rows):
 *   out = v_scale * sum_t e^(s_t) v_t / (sum_t e^(s_t) + e^(sinks[h]))
 *   lse = ln(sum_t e^(s_t) + e^(sinks[h]))
 * A sink of -inf leaves the head unchanged. sinks must not be NULL; the
 * other arguments are those of paged_decode_run.
 */
pd_status paged_decode_run_sinks(const pd_plan* plan, const void* q, const void* k_pool,
                                 const void* v_pool, const int32_t* block_tables,
                                 const int32_t* seq_lens, const int32_t* q_indptr, float sm_scale,
                                 const float* k_scale, const float* v_scale, const float* sinks,
                                 void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 pd_stream_t stream);

/*
 * Paged prefill / context attention (problem->kind == PD_ATTN_PREFILL): the
 * context call of the cake_fmha API page (trtllm_batch_context_with_kv_cache,
 * the same arguments as the decode call), for requests with many new tokens.
 * It computes exactly what paged_decode_run computes (inclusive causal bound
 * pos = seq_lens[b] - q_len_b + i), with two 128-row tiles of packed (token, head) query rows
 * and 128 keys per tensor-core tile.
 *   q, k_pool, v_pool, block_tables, seq_lens, q_indptr, out, lse,
 *   workspace: as for paged_decode_run, BF16 pools only
 *   sm_scale finite and > 0 (PD_ERR_INVALID_ARG otherwise)
 *   sinks    NULL or device fp32 [Hq] (as for paged_decode_run_sinks)
 * The plan must have head_dim 128, kv_dtype PD_KV_BF16, a page size that is
 * a multiple of 8 and a group Hq / Hkv that divides 128 (paged_decode_plan
 * returns PD_ERR_UNSUPPORTED otherwise). Split units are merged by the
 * LSE-merge kernel (the plan's merge mode is PD_MERGE_KERNEL).
 */
pd_status paged_prefill_run(const pd_plan* plan, const void* q, const void* k_pool,
                            const void* v_pool, const int32_t* block_tables,
                            const int32_t* seq_lens, const int32_t* q_indptr, float sm_scale,
                            const float* sinks, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, pd_stream_t stream);

/*
 * MLA decode (problem->kind == PD_ATTN_MLA): one latent KV head shared by
 * every query head.
 *   q        bf16 [total_q][H][576]
 *   kv_pool  bf16 [num_pages][P][576] (page stride k_page_stride)
 *   out      bf16 [total_q][H][512];  lse fp32 [total_q][H] or NULL
 * Other arguments as for paged_decode_run. The page size must be a multiple
 * of 8 (paged_decode_plan returns PD_ERR_UNSUPPORTED otherwise).
 */
pd_status mla_decode_run(const pd_plan* plan, const void* q, const void* kv_pool,
                         const int32_t* block_tables, const int32_t* seq_lens,
                         const int32_t* q_indptr, float sm_scale, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, pd_stream_t stream);

/* mla_decode_run with attention sinks (device fp32 [H], as for
 * paged_decode_run_sinks; not NULL). */
pd_status mla_decode_run_sinks(const pd_plan* plan, const void* q, const void* kv_pool,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* q_indptr, float sm_scale, const float* sinks,
                               void* out, float* lse, void* workspace, size_t workspace_bytes,
                               pd_stream_t stream);

/*
 * FP8 latent MLA (PR #5552 "Kimi-K3 FP8 latent MLA": FP8 query and FP8
 * latent cache): the plan's kv_dtype is PD_KV_FP8_E4M3 and both the query
 * and the pool hold OCP E4M3 codes.
 *   q        e4m3 [total_q][H][576], value = code * q_scale[0]
 *   kv_pool  e4m3 [num_pages][P][576] (page stride k_page_stride, bytes),
 *            value = code * kv_scale[0]; key = the row, value = channels 0..511
 *   q_scale, kv_scale  device fp32 scalars (required)
 *   sinks    NULL or device fp32 [H] (as for mla_decode_run_sinks)
 *   out      bf16 [total_q][H][512];  lse fp32 [total_q][H] or NULL
 * The kernel multiplies E4M3 operands on the tensor cores (fp32
 * accumulation) and rounds the softmax probabilities to E4M3 for the P.V
 * product (as the pages' FP8 programs do; accuracy: the E4M3 tolerance).
 */
pd_status mla_decode_run_fp8(const pd_plan* plan, const void* q, const void* kv_pool,
                             const int32_t* block_tables, const int32_t* seq_lens,
                             const int32_t* q_indptr, float sm_scale, const float* q_scale,
                             const float* kv_scale, const float* sinks, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, pd_stream_t stream);

/*
 * Paged KV append: writes the K and V rows of the new tokens into the pools,
 * the step before decode (PR #5952 "fused BF16 QK RMSNorm + NeoX RoPE + paged
 * KV append", commit #5956 "Contract"; the fused RMSNorm / RoPE of that PR
 * are not part of this call). seq_lens is the total length after the append,
 * so new token i of request b (rows q_indptr[b] .. q_indptr[b+1]-1 of the new
 * rows) goes to position seq_lens[b] - n_b + i: page
 * block_tables[b][pos / page_size], slot pos % page_size.
 *   k_new, v_new  bf16 [total_new][num_kv_heads][head_dim], 8-byte aligned
 *                 (when both are 16-byte aligned they are read in 16-byte
 *                 chunks, the faster path; the results are the same);
 *                 v_new and v_pool may both be NULL for a K-only pool (the
 *                 MLA latent cache: num_kv_heads 1, head_dim 576, NHD)
 *   k_pool, v_pool the pools of prob->layout and prob->kv_dtype (16-byte
 *                 aligned); BF16 pools receive the bits; E4M3 pools receive
 *                 x / scale (binary32 quotient) rounded to nearest even and
 *                 saturated to +-448, with k_scale / v_scale device fp32
 *                 scalars, positive and finite (required for E4M3, ignored
 *                 for BF16)
 *   zero_tail     nonzero: the slots of each request's last page past
 *                 seq_lens[b] are zeroed as well (K and V)
 *   error_word    NULL or a device int32[2] (code, request) that receives the
 *                 first pd_device_error: PD_DEV_BAD_PAGE for a page id outside
 *                 [0, num_pages) (that row is not written),
 *                 PD_DEV_SEQ_LEN_MISMATCH for n_b > seq_lens[b] (the request
 *                 is not written), PD_DEV_Q_INDPTR_MISMATCH when total_new
 *                 exceeds q_indptr[batch]. The caller zeroes it.
 * head_dim must be a multiple of 8 and at most 1024; page strides (elements,
 * 0 = compact) must be multiples of 16 bytes. Asynchronous on `stream`; no
 * allocation; total_new = 0 with zero_tail = 0 is a no-op.
 */
typedef struct {
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages_per_seq;  /* row length of block_tables                 */
  int32_t layout;             /* pd_layout                                   */
  int32_t kv_dtype;           /* pd_kv_dtype                                 */
  int64_t k_page_stride;      /* elements; 0 = compact (P * Hkv * head_dim)  */
  int64_t v_page_stride;
} pd_append_problem;

pd_status paged_kv_append(const pd_append_problem* prob, const void* k_new, const void* v_new,
                          int32_t total_new, const int32_t* q_indptr, const int32_t* seq_lens,
                          const int32_t* block_tables, const float* k_scale, const float* v_scale,
                          void* k_pool, void* v_pool, int32_t zero_tail, int32_t* error_word,
                          pd_stream_t stream);

/*
 * LSE merge of attention states over disjoint key ranges (the split-KV
 * combine step as a kernel of its own):
 *   v_states fp32 [num_states][rows][dim] normalised partial outputs
 *   s_states fp32 [num_states][rows]      their natural-log LSE (-inf = empty)
 *   out      bf16 [rows][dim] = sum_s exp(s_s - lse) v_s
 *   lse_out  fp32 [rows] = log sum_s exp(s_s), or NULL
 * 1 <= num_states <= 64, dim a multiple of 8 and <= 1024. Rows whose
 * states are all empty give out = 0, lse = -inf.
 */
pd_status paged_decode_merge_states(const float* v_states, const float* s_states,
                                    int32_t num_states, int64_t rows, int32_t dim, void* out,
                                    float* lse_out, pd_stream_t stream);

/*
 * Allocation-free variant of paged_decode_run. (The pages have no
 * counterpart: this entry point exists for callers of this library that may
 * not allocate device memory, e.g. a runtime that reserves all device memory
 * at start-up and forbids later cudaMalloc calls, or a plugin whose host
 * framework owns the allocator.)
 *
 * The workspace is a fixed array of PD_NO_ALLOC_MAX_WORKSPACE_BYTES bytes in
 * the library's own device memory, present on every GPU that loads the
 * library until the process exits. Each call copies the plan into it (one
 * host-to-device copy on `stream`, which also zeroes the split counters and
 * the error word) and then runs exactly as paged_decode_run; the caller
 * passes inputs and outputs as for that call. Nothing is allocated.
 *  - Plans whose paged_decode_workspace_size exceeds
 *    PD_NO_ALLOC_MAX_WORKSPACE_BYTES are refused with
 *    PD_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - The first call on a device looks up the array's device address with that
 *    device current and caches it. The cached address belongs to the
 *    runtime's primary context:
 *    do not call cudaDeviceReset between calls, and do not call this entry
 *    point under another driver context of the device.
 *  - Every call on a device shares the one array: calls whose work can
 *    overlap on the GPU (other streams, other host threads) race and must be
 *    serialised by the caller. The array keeps the last call's contents.
 *  - Device-side errors are reported in the array's error word, which this
 *    entry point does not expose; check results with paged_decode_run when
 *    diagnosing.
 */
#define PD_NO_ALLOC_MAX_WORKSPACE_BYTES ((size_t)32 << 20)
pd_status paged_decode_run_no_alloc(const pd_plan* plan, const void* q, const void* k_pool,
                                    const void* v_pool, const int32_t* block_tables,
                                    const int32_t* seq_lens, const int32_t* q_indptr,
                                    float sm_scale, const float* k_scale, const float* v_scale,
                                    void* out, float* lse, pd_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the workspace's device error
 * word. *code_out gets a pd_device_error, *info_out the request index (or
 * -1). Returns PD_ERR_DEVICE_FLAG when the code is not PD_DEV_OK.
 */
pd_status paged_decode_read_error(void* workspace, int32_t* code_out, int32_t* info_out,
                                  pd_stream_t stream);

void paged_decode_plan_destroy(pd_plan* plan);

const char* pd_status_string(pd_status status);

/* Text of the CUDA error behind the calling thread's last PD_ERR_CUDA
 * (empty if none); valid until that thread's next library call. */
const char* paged_decode_last_cuda_error(void);

/*
 * Limit, in nanoseconds, of every pipeline wait inside the kernels that are
 * launched after this call, process-wide (0 restores the default of 2 s).
 * A wait that runs past it ends its kernel early with PD_DEV_TIMEOUT in the
 * workspace error word (paged_decode_read_error) instead of waiting on; each
 * CTA first drains its own copies and tensor-core work, so the context stays
 * usable. The outputs of that call are then undefined, and the workspace must
 * be uploaded again (paged_decode_plan_upload) before its next run, since
 * split counters may be left mid-count. No wait gives up in less than about
 * 20 us. Meant for exercising the failure path; the default suits any call.
 */
pd_status paged_decode_set_wait_limit_ns(uint64_t limit_ns);

/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t paged_decode_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_DECODE_H */
