/*
 * ekv.h -- C ABI of the ekv library: mixed-fidelity paged KV attention on GB300.
 *
 * Three operations, from the pages' statement of the problem:
 *
 *  - ekv_paged_decode: paged GQA decode attention that reads the mixed-fidelity KV
 *    cache directly. Keys are FP16; each value page is TARGET (FP16) or compact
 *    (FP8 E4M3 codes times a scale). ElasticKV ("Does Execution Require Target KV
 *    Fidelity?"), Sec. 3.2 "Dual-mode Elastic Attention Backend": both fidelities are
 *    consumed directly behind one attention interface, the compact state is expanded
 *    in registers and never materialised, and TARGET-only batches keep the native
 *    path. knlp.io "Asymmetric K16/V8 KV cache", Fig. "Fresh prefill gets a fast path
 *    inside a mixed batch": the decode prefix reads persistent FP16 keys and FP8
 *    values, and existing value scales still apply in attention.
 *  - ekv_gather_prefill: compact prefill gathers stored K16/V8 pages into one bounded
 *    FP16 workspace for a native FP16 prefill, casting V8 -> FP16 (knlp.io, "What
 *    changes in vLLM's prefill routing?"; at most 4,096 pages, 256 MiB payload).
 *  - ekv_demote_pages: TARGET -> compact demotion, synchronous and in place on the
 *    GPU, the new state visible only after completion (ElasticKV Sec. 3.4
 *    "Transition protocols"), requantising FP16 value pages to E4M3 with one absmax
 *    scale per (page, KV head).
 *
 * Conventions for every entry point:
 *  - Data pointers are DEVICE pointers owned by the caller, unless stated otherwise.
 *    The library never frees or keeps them beyond the call.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Work is enqueued on it
 *    and the call returns without synchronising. Hot calls allocate nothing.
 *  - Argument errors are found on the host and returned before anything is launched.
 *  - Errors found by the kernels (a page id outside the pool, a non-finite or <= 0
 *    scale, a seq_len above the block table's capacity, a demotion page holding
 *    NaN/inf, a timed-out pipeline wait) set a sticky error word in the context; the
 *    affected outputs are zeroed (decode) or left untouched (demote). Read and clear it
 *    with ekv_get_error. In decode, a page that fails its check zeroes the output (and
 *    sets lse = -inf) of the query heads that read it: the whole sequence for a bad
 *    page id or mode byte, the G query heads of one KV head for a bad per-(page, head)
 *    scale; a sequence whose seq_len fails is written as empty.
 *  - A context is bound to the device current at ekv_create and to one stream at a
 *    time: calls that overlap on different streams race on its scratch.
 *
 * Page layout (NHD, page size 16, knlp.io measured route: "NHD layout, page size 16"):
 *  - K pool: fp16 [num_pages][16][H_kv][D], contiguous.
 *  - V pool: bytes [num_pages][v_page_stride_bytes]. A TARGET page holds fp16
 *    [16][H_kv][D] in its first 16*H_kv*D*2 bytes; a compact page holds E4M3 codes
 *    [16][H_kv][D] in its first 16*H_kv*D bytes. A uniform compact pool may use
 *    stride 16*H_kv*D; a pool that holds TARGET pages needs stride >= 16*H_kv*D*2.
 *    The stride must be a multiple of 16 bytes.
 *  - Supported: H_kv in {1,2,4,8}, G = H_q/H_kv in {1..8}, D in {64,128}.
 */
#ifndef EKV_H
#define EKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EKV_OK = 0,
  EKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size/stride/enum, misaligned pointer */
  EKV_ERR_UNSUPPORTED = 2,   /* shape outside the supported set: take your existing path */
  EKV_ERR_CAPACITY = 3,      /* more pages than the workspace / context was sized for */
  EKV_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, allocation, ...) */
  EKV_ERR_DEVICE_CHECK = 5   /* a kernel found bad data (see ekv_get_error detail) */
} ekv_status;

/* Per-page value fidelity, one uint8 per physical page.
 *  TARGET_FP16:   the page's value slot holds fp16 [16][H_kv][D].
 *  COMPACT_E4M3:  its first 16*H_kv*D bytes are E4M3 codes; value = E4M3(code) * scale
 *                 (knlp.io "Asymmetric K16/V8 KV cache").
 *  BASE:          its first 16*H_kv*D bytes are the high bytes of the fp16 values; value =
 *                 the fp16 whose high byte is the stored byte and whose low byte is zero,
 *                 no scale (ElasticKV Sec. 3.2 and App. B.3: "shift-and-bitcast"). The low
 *                 bytes, kept by the caller, restore TARGET exactly (ekv_promote_pages). */
typedef enum { EKV_MODE_TARGET_FP16 = 0, EKV_MODE_COMPACT_E4M3 = 1, EKV_MODE_BASE = 2 } ekv_page_mode;

/* Granularity of the compact-page value scales (fp32, device memory).
 * PER_TENSOR: v_scales[0] applies to every compact page (a per-layer scale is one
 * per-tensor scale per call). PER_PAGE_HEAD: v_scales[p * H_kv + h]. */
typedef enum { EKV_SCALE_PER_TENSOR = 0, EKV_SCALE_PER_PAGE_HEAD = 1 } ekv_scale_mode;

/* Detail codes reported with EKV_ERR_DEVICE_CHECK by ekv_get_error. */
typedef enum {
  EKV_DETAIL_NONE = 0,
  EKV_DETAIL_PAGE_ID = 1,        /* block_table / page_ids entry outside [0, num_pages) */
  EKV_DETAIL_SCALE = 2,          /* a scale read by a compact page is NaN, inf or <= 0 */
  EKV_DETAIL_SEQ_LEN = 3,        /* seq_lens[b] < 0 or > block_table_stride * 16 */
  EKV_DETAIL_NONFINITE_PAGE = 4, /* a page given to demotion holds NaN or inf */
  EKV_DETAIL_TIMEOUT = 5,        /* a bounded pipeline wait gave up */
  EKV_DETAIL_PAGE_MODE = 6       /* a page_mode byte is not TARGET, COMPACT or BASE */
} ekv_detail;

typedef struct ekv_ctx ekv_ctx;

typedef struct {
  int num_q_heads;        /* H_q */
  int num_kv_heads;       /* H_kv; H_q % H_kv == 0 */
  int head_dim;           /* D: 64 or 128 */
  int max_batch;          /* largest `batch` a decode call may pass (sizes the scratch) */
} ekv_config;

/* Create a context on the current device: allocates the split-K partials, the plan
 * buffer and the sticky error word once (cudaMalloc). Returns EKV_ERR_UNSUPPORTED for
 * shapes outside the supported set. *ctx is NULL on failure. */
ekv_status ekv_create(ekv_ctx** ctx, const ekv_config* cfg);

/* Free the context's device memory (synchronises the device first). NULL is a no-op. */
ekv_status ekv_destroy(ekv_ctx* ctx);

/* Paged GQA decode attention: for every sequence b and query head h_q,
 *   out[b][h_q] = sum_t softmax_t(sm_scale * q[b][h_q] . k_t) v_t
 * over the seq_lens[b] tokens of b, token t at page block_table[b][t/16], row t%16,
 * KV head h_q / G; v_t is the FP16 row of a TARGET page or E4M3(code) * scale of a
 * compact page. One query per sequence attends to all its cached tokens (no mask).
 *
 *  q            fp16 [batch][H_q][D], contiguous.
 *  k_pages      fp16 [num_pages][16][H_kv][D]; 16-byte aligned.
 *  v_pages      bytes [num_pages][v_page_stride_bytes]; 16-byte aligned.
 *  v_scales     fp32, see ekv_scale_mode; may be NULL only if no page is compact.
 *  page_mode    uint8 [num_pages] or NULL; NULL means every page has `uniform_mode`
 *               (the uniform paths load no mode bytes; uniform TARGET loads no scales).
 *  block_table  int32 [batch][block_table_stride]; entries past a sequence's pages
 *               are not read.
 *  seq_lens     int32 [batch]; 0 gives out = 0 and lse = -inf.
 *  sm_scale     softmax scale; <= 0 means 1/sqrt(D).
 *  out          fp16 [batch][H_q][D] (written).
 *  lse          fp32 [batch][H_q] natural-log log-sum-exp of the scaled scores, or NULL.
 * Returns EKV_ERR_CAPACITY when batch > cfg.max_batch. */
ekv_status ekv_paged_decode(ekv_ctx* ctx, const void* q, const void* k_pages,
                            const void* v_pages, long long v_page_stride_bytes,
                            int num_pages, const float* v_scales, int scale_mode,
                            const uint8_t* page_mode, int uniform_mode,
                            const int32_t* block_table, int block_table_stride,
                            const int32_t* seq_lens, int batch, float sm_scale,
                            void* out, float* lse, void* stream);

/* Paged decode over ElasticKV's pair-structured value layout (ElasticKV Sec. 3.1 "Pair-
 * Structured Elastic KV Layout", Sec. 3.2, App. B.3). Same computation as
 * ekv_paged_decode; the values of logical page p (keys and mode byte stay at p) are
 * found through a separate value block table, so two compact or BASE pages can share
 * one physical value slot and free the other for the allocator.
 *  v_pages        bytes [num_v_slots][v_page_stride_bytes], stride >= 32*H_kv*D: each slot
 *                 holds one TARGET page or two halves of 16*H_kv*D bytes.
 *  v_block_table  int32 [batch][block_table_stride]: value location of logical page j of
 *                 sequence b, a half-slot index e in [0, 2*num_v_slots): a TARGET page fills
 *                 slot e/2 (e must be even); a compact or BASE page is half e%2 of slot e/2.
 *  boundaries     int32 [batch][2] or NULL: ElasticKV's structured TARGET-BASE-TARGET
 *                 layout, pages boundaries[b][0] <= j < boundaries[b][1] of sequence b are
 *                 BASE and the others TARGET; no mode byte is read. NULL: page_mode (by
 *                 logical page) or uniform_mode, as in ekv_paged_decode.
 *  has_base       0: the batch holds TARGET pages only and runs the native FP16 path
 *                 (ElasticKV's batch-level BASE indicator); modes and boundaries are not
 *                 read. Nonzero: the elastic path.
 * A location outside the pool, or an odd one for a TARGET page, is a device error
 * (EKV_DETAIL_PAGE_ID) that zeroes the heads that read it. Other arguments as for
 * ekv_paged_decode. */
ekv_status ekv_paged_decode_elastic(ekv_ctx* ctx, const void* q, const void* k_pages,
                                    const void* v_pages, long long v_page_stride_bytes,
                                    int num_pages, int num_v_slots, const float* v_scales,
                                    int scale_mode, const uint8_t* page_mode, int uniform_mode,
                                    const int32_t* block_table, const int32_t* v_block_table,
                                    int block_table_stride, const int32_t* boundaries,
                                    int has_base, const int32_t* seq_lens, int batch,
                                    float sm_scale, void* out, float* lse, void* stream);

/* Compact-prefill gather: copies the pages named by `page_range` into consecutive
 * workspace slots, in page_range order.
 *
 *  page_range   HOST int32 [n][3] rows {seq, first_page, num_pages}: logical pages
 *               first_page .. first_page+num_pages-1 of sequence `seq`, reached through
 *               block_table[seq]. 0 <= seq < block_table_rows and
 *               first_page + num_pages <= block_table_stride are checked on the host.
 *  ws_k, ws_v   fp16 [ws_pages][16][H_kv][D]: ws_k[w] = K page bit for bit; ws_v[w] =
 *               the TARGET page bit for bit, or fp16_rn(fp32_rn(E4M3(code) * scale))
 *               for a compact page (fp16(E4M3(code)) when apply_scale == 0).
 *  ws_indices   int32 [ws_pages]: ws_indices[w] = w for every gathered page, the
 *               workspace page table an FP16 prefill reads.
 * Returns EKV_ERR_CAPACITY when the total page count exceeds ws_pages (nothing is
 * launched). Other layout arguments are as for ekv_paged_decode. */
ekv_status ekv_gather_prefill(ekv_ctx* ctx, const void* k_pages, const void* v_pages,
                              long long v_page_stride_bytes, int num_pages,
                              const float* v_scales, int scale_mode,
                              const uint8_t* page_mode, int uniform_mode,
                              const int32_t* block_table, int block_table_stride,
                              int block_table_rows, const int32_t* page_range, int n,
                              void* ws_k, void* ws_v, int32_t* ws_indices, int ws_pages,
                              int apply_scale, void* stream);

/* The compact-prefill gather from ElasticKV's pair-structured value layout (ElasticKV
 * Sec. 3.1, Sec. 3.2): as ekv_gather_prefill, but the values of logical page j of
 * sequence b are read at half-slot location v_block_table[b][j] (a TARGET page fills slot
 * e/2, e even; a compact or BASE page is half e%2 of slot e/2), and a page's mode comes
 * from boundaries (T-B-T: BASE for boundaries[b][0] <= j < boundaries[b][1]), else from
 * page_mode / uniform_mode; has_base = 0 gathers every page as TARGET. Keys stay at the
 * logical page. v_pages, num_v_slots, v_block_table, boundaries and has_base as for
 * ekv_paged_decode_elastic (v_block_table must not be NULL). A location outside the pool,
 * or an odd one for a TARGET page, is a device error (EKV_DETAIL_PAGE_ID) that zeroes the
 * workspace page. */
ekv_status ekv_gather_prefill_elastic(ekv_ctx* ctx, const void* k_pages, const void* v_pages,
                                      long long v_page_stride_bytes, int num_pages, int num_v_slots,
                                      const float* v_scales, int scale_mode,
                                      const uint8_t* page_mode, int uniform_mode,
                                      const int32_t* block_table, const int32_t* v_block_table,
                                      int block_table_stride, const int32_t* boundaries,
                                      int has_base, int block_table_rows,
                                      const int32_t* page_range, int n, void* ws_k, void* ws_v,
                                      int32_t* ws_indices, int ws_pages, int apply_scale,
                                      void* stream);

/* FP16 causal prefill of whole prompts over the gathered workspace (knlp.io "What
 * changes in vLLM's prefill routing?": after the gather casts the stored K16/V8 pages into
 * the bounded FP16 workspace, a native FP16 prefill runs over it; causal, no cached
 * prefix, no sliding window). For prompt i with len_i = cu_seqlens[i+1] - cu_seqlens[i]
 * tokens, query position s (row cu_seqlens[i] + s of q) and query head h_q:
 *   out = sum_{t <= s} softmax_t(sm_scale * q . k_t) v_t,  k_t / v_t = row t % 16 of
 *   workspace page page_off[i] + t / 16, KV head h_q / G;  lse = log sum e^(...).
 *  q, out       fp16 [T][H_q][D], T = cu_seqlens[n]; 16-byte aligned.
 *  ws_k, ws_v   fp16 [ws_pages][16][H_kv][D] (the gather's workspace), 16-byte aligned.
 *  cu_seqlens   DEVICE int32 [n + 1], nondecreasing; page_off DEVICE int32 [n].
 *  max_len      HOST int >= every len_i (sizes the grid); a longer prompt is reported
 *               (EKV_DETAIL_SEQ_LEN): its first max_len rows are computed (causal rows
 *               need no later key) and its later rows are not written.
 *  lse          fp32 [T][H_q] (natural log) or NULL.
 * A prompt whose pages fall outside [0, ws_pages) is reported (EKV_DETAIL_PAGE_ID). */
ekv_status ekv_prefill_attention(ekv_ctx* ctx, const void* q, const void* ws_k, const void* ws_v,
                                 int ws_pages, const int32_t* cu_seqlens, const int32_t* page_off,
                                 int n, int max_len, float sm_scale, void* out, float* lse,
                                 void* stream);

/* TARGET -> compact demotion, in place. For each page p = page_ids[i] whose
 * page_mode[p] is TARGET, and each KV head h:
 *   a = max |x| over the page's 16 x D fp16 values of head h,
 *   s = fp32_rn(a / 448) (1.0 when a == 0),  code = E4M3_rn_satfinite(fp32_rn(x / s)),
 * writes the codes into the first 16*H_kv*D bytes of the page's value slot,
 * scale_out[p * H_kv + h] = s, then page_mode[p] = COMPACT. Pages that are not TARGET
 * are skipped; a page holding NaN/inf is left TARGET and reported
 * (EKV_DETAIL_NONFINITE_PAGE).
 *  v_pages      bytes [num_pages][v_page_stride_bytes], stride >= 16*H_kv*D*2.
 *  page_ids     int32 [n], distinct (duplicates race on the same page).
 *  page_mode    uint8 [num_pages] (read and written).
 *  scale_out    fp32 [num_pages][H_kv] (written for demoted pages).
 * No decode or gather may read these pages concurrently on another stream. */
ekv_status ekv_demote_pages(ekv_ctx* ctx, void* v_pages, long long v_page_stride_bytes,
                            int num_pages, const int32_t* page_ids, int n,
                            uint8_t* page_mode, float* scale_out, void* stream);

/* TARGET -> BASE demotion, in place (ElasticKV Sec. 3.4 "Transition protocols",
 * App. B.2). For each page p = page_ids[i] whose page_mode[p] is TARGET: the high
 * byte of every fp16 value of the page goes to the first 16*H_kv*D bytes of its value
 * slot (same element order), the low bytes to row i of low_out, then page_mode[p] =
 * BASE. Pages that are not TARGET are skipped (their row untouched); a page holding
 * NaN/inf is left TARGET and reported (EKV_DETAIL_NONFINITE_PAGE).
 *  low_out      bytes [n][16*H_kv*D], 16-byte aligned, or NULL to drop the low bytes
 *               (the page can then not be promoted exactly). Device memory, or host
 *               memory the device can address (mapped pinned memory): ElasticKV keeps
 *               this refinement in CPU backing.
 * Other arguments as for ekv_demote_pages. */
ekv_status ekv_demote_pages_base(ekv_ctx* ctx, void* v_pages, long long v_page_stride_bytes,
                                 int num_pages, const int32_t* page_ids, int n,
                                 uint8_t* page_mode, void* low_out, void* stream);

/* BASE -> TARGET promotion, in place and exact (ElasticKV App. B.2: one step from the
 * 8-bit BASE state back to the original 16-bit TARGET). For each page p = page_ids[i]
 * whose page_mode[p] is BASE: value = (high byte << 8) | low_in[i][e] for every element
 * e, written as fp16 over the page's value slot, then page_mode[p] = TARGET. Pages
 * that are not BASE are skipped.
 *  low_in       bytes [n][16*H_kv*D], 16-byte aligned (the rows ekv_demote_pages_base
 *               wrote, in the order of this call's page_ids); device or mapped host
 *               memory.
 * The new mode is visible in stream order, after the call's work completes; no decode
 * or gather may read these pages concurrently on another stream. */
ekv_status ekv_promote_pages(ekv_ctx* ctx, void* v_pages, long long v_page_stride_bytes,
                             int num_pages, const int32_t* page_ids, int n,
                             uint8_t* page_mode, const void* low_in, void* stream);

/* Page-mode transitions with value locations (ElasticKV Sec. 3.1 and App. B.2), the
 * general form of ekv_demote_pages (op 0), ekv_demote_pages_base (op 1) and
 * ekv_promote_pages (op 2) for the layout of ekv_paged_decode_elastic. Item i concerns
 * logical page page_ids[i] (its page_mode byte, and for op 0 its scale_out row):
 *  op 0 / 1     reads the TARGET page at the even location src_loc[i] (its whole slot) and
 *               writes its E4M3 codes / BASE high bytes to the half at dst_loc[i];
 *  op 2         reads the BASE half at src_loc[i] and the low bytes low[i], writes the TARGET
 *               page over the slot of the even location dst_loc[i].
 * src_loc / dst_loc NULL mean in place (2 * page_ids[i]). Items of one call run
 * concurrently: no item may write a location another item of the call reads. Packing a
 * pair (A, B) into A's slot therefore takes two calls: A in place, then B from its slot
 * to half 1 of A's slot; B's slot is then free.
 *  low          op 1: bytes [n][16*H_kv*D] out (may be NULL); op 2: in (required).
 *  num_slots    value slots of v_pages; num_pages: logical pages (page_mode, scale_out).
 * Skips, checks and errors as for the three calls above; a location outside the pool,
 * or an odd one where a TARGET page is read or written, is reported (EKV_DETAIL_PAGE_ID)
 * and its item skipped. */
ekv_status ekv_transition_pages(ekv_ctx* ctx, int op, void* v_pages, long long v_page_stride_bytes,
                                int num_slots, int num_pages, const int32_t* page_ids,
                                const int32_t* src_loc, const int32_t* dst_loc, int n,
                                uint8_t* page_mode, float* scale_out, void* low, void* stream);

/* K16/V8 cache writer: stores one new token per sequence into the paged cache
 * (knlp.io "Asymmetric K16/V8 KV cache", implementation checks: "vLLM cache writer: K
 * bit-exact, V within FP8 noise"). For each b with t = positions[b] >= 0, the token goes
 * to row t % 16 of page p = block_table[b][t / 16]:
 *   K row = k_new[b] (fp16 bits);
 *   V row, by page_mode[p] (or uniform_mode): TARGET = v_new[b] (fp16 bits); COMPACT_E4M3 =
 *   E4M3_rn_satfinite(fp32_rn(v / s)) with the page's existing scale s (per tensor or
 *   per (p, KV head)); BASE = the high bytes of v_new[b].
 * The caller allocates pages and grows seq_lens (to t + 1) itself; the first token of a
 * page is written into a page whose other rows are not read until later steps fill them.
 *  k_new, v_new  fp16 [batch][H_kv][D], 16-byte aligned.
 *  positions     int32 [batch]; < 0 means no token for that sequence this step.
 * Device checks (reported, nothing written for that sequence): t >= block_table_stride *
 * 16 (EKV_DETAIL_SEQ_LEN), a page id outside the pool, a mode byte > 2. A compact page
 * whose scale for a KV head is missing or not positive finite keeps that head's old
 * bytes (EKV_DETAIL_SCALE). Other arguments as for ekv_paged_decode. */
ekv_status ekv_append_kv(ekv_ctx* ctx, const void* k_new, const void* v_new, void* k_pages,
                         void* v_pages, long long v_page_stride_bytes, int num_pages,
                         const float* v_scales, int scale_mode, const uint8_t* page_mode,
                         int uniform_mode, const int32_t* block_table, int block_table_stride,
                         const int32_t* positions, int batch, void* stream);

/* Paged decode that allocates nothing, for callers that must not call cudaMalloc on
 * this path (a runtime whose pool owns all device memory, an enqueue hook of a host
 * framework that forbids allocation, a fixed start-up memory budget). The pages have
 * no counterpart of this call: it computes exactly what ekv_paged_decode computes, for
 * the shape given in its first three arguments, without a context.
 *
 * Its split-K scratch (partial records, tickets, error word) is one 16 MiB array of
 * device memory compiled into the library: every GPU that loads the library holds it
 * until the process exits. The first 128 KiB hold the tickets (4,096 x 8 ints), then
 * 256 B of error word, then the records, aligned to 256 B: (batch + #SMs) * (8 / H_kv)
 * * H_q float2 (m, l) pairs and as many * D floats must fit in what is left; a call
 * whose records need more returns EKV_ERR_CAPACITY (batch <= 4096).
 *  - The first call on a device looks up the array's device address (and the SM
 *    count) with that device current; make that first call before any stream capture.
 *    The address stays valid for the life of the device's primary context: do not use
 *    this entry point on a device after cudaDeviceReset (the address looked up before
 *    the reset would then be stale).
 *  - Every call shares the one array and starts by clearing its tickets on `stream`:
 *    calls that overlap on the GPU (other streams, other host threads) race on it.
 *  - err_out: device int[4] that receives {ekv_status, ekv_detail, index, 0} of the
 *    first data error the kernel finds (zeroed by the call first), or NULL.
 * No cudaMalloc, cudaFree or allocating library call is made; work is enqueued on
 * `stream` (cudaMemsetAsync of the tickets and err_out, then one kernel launch). The
 * other arguments and all layouts are those of ekv_paged_decode. */
ekv_status ekv_paged_decode_noalloc(int num_q_heads, int num_kv_heads, int head_dim,
                                    const void* q, const void* k_pages, const void* v_pages,
                                    long long v_page_stride_bytes, int num_pages,
                                    const float* v_scales, int scale_mode,
                                    const uint8_t* page_mode, int uniform_mode,
                                    const int32_t* block_table, int block_table_stride,
                                    const int32_t* seq_lens, int batch, float sm_scale,
                                    void* out, float* lse, int* err_out, void* stream);

/* Synchronise the stream of the context's last call (that stream only), read the
 * sticky device error word and clear it; after an error the context's ticket buffer is
 * cleared too, so a call that wound down early leaves nothing behind for the next one.
 * *code is an ekv_status (EKV_OK or EKV_ERR_DEVICE_CHECK), *detail an ekv_detail. Either
 * pointer may be NULL. Returns EKV_ERR_CUDA if the sync fails. After EKV_DETAIL_TIMEOUT
 * the outputs of the call that reported it are undefined. */
ekv_status ekv_get_error(ekv_ctx* ctx, int* code, int* detail);

/* Kernel timing for measurement: when enabled, each ekv_paged_decode records CUDA
 * events around its split-K kernel on the launching stream. ekv_profile_read
 * synchronises, returns the summed split-kernel time in milliseconds and the number
 * of timed launches since the last read, and resets both. */
ekv_status ekv_profile_enable(ekv_ctx* ctx, int enable);
ekv_status ekv_profile_read(ekv_ctx* ctx, double* split_ms, long long* launches);

/* The fixed cost of one timed launch, for reading the split-kernel times above: `reps`
 * (1..1024) launches of an empty kernel with the split kernel's grid, block, dynamic
 * shared memory (D = head_dim, E4M3 slots) and parameter size, each between two CUDA
 * events on `stream` (NULL = the default stream) exactly as a profiled decode is. Writes
 * the average milliseconds between the two events of one launch to *avg_ms. The kernel
 * touches no memory. Synchronises the stream; EKV_ERR_CUDA on a CUDA failure. */
ekv_status ekv_profile_launch_floor(ekv_ctx* ctx, int reps, void* stream, double* avg_ms);

/* Consumer variant of this context. Decode: 0 (default) multiplies the QK and PV
 * tiles on the tensor cores (mma.sync f16 -> f32); 1 uses CUDA-core FP32 FMAs. Prefill
 * (ekv_prefill_attention): 0 runs on the fifth-generation tensor cores (tcgen05 MMA,
 * tensor-memory accumulators, TMA loads), 1 on warp-level mma.sync. Both variants
 * compute the same function; 1 exists for measurement. */
ekv_status ekv_set_decode_variant(ekv_ctx* ctx, int variant);

/* Programmatic dependent launch (CUDA's griddepcontrol, sm_90+) of the decode and the
 * gather, for streams of back-to-back calls (a decode per layer; the gather chunks of a
 * prefill admission). enable = 1: ekv_paged_decode, ekv_paged_decode_elastic (decode
 * variant 0), ekv_gather_prefill and ekv_gather_prefill_elastic are launched with
 * programmatic stream serialization and signal their own dependents at kernel start,
 * so the next call's first reads run on SMs as this call's CTAs leave.
 * What CUDA guarantees, and therefore the contract: a kernel launched this way may
 * start before the kernel ahead of it in the stream (the "primary") has finished, and
 * the primary's memory writes are guaranteed visible to it only after its
 * grid-dependency wait (CUDA C++ Programming Guide, "Programmatic Dependent Launch and
 * Synchronization": cudaGridDependencySynchronize / griddepcontrol.wait).
 *  - Before that wait the decode reads seq_lens, the block tables, page_mode, v_scales,
 *    boundaries and the K/V pages that are not the last page of their sequence; it
 *    reads q and writes out, lse and its workspace after the wait. The kernel
 *    immediately ahead of a decode may therefore write q and the last page of each
 *    sequence (ekv_append_kv does exactly that) but none of the other inputs.
 *  - Before that wait the gather reads the block tables, page_mode, v_scales,
 *    boundaries and every K/V page it copies; it writes the workspace, the indices and
 *    the error word after the wait. The kernel immediately ahead of a gather may write
 *    none of its inputs.
 * The library keeps these rules for its own kernels: the page-mode transitions
 * (ekv_demote_pages, ekv_demote_pages_base, ekv_promote_pages, ekv_transition_pages)
 * write value pages, mode bytes and scales, and ekv_append_kv writes pool pages, so a
 * decode enqueued on a stream whose last kernel from this library (any context) is a
 * transition, and a gather whose last such kernel is a transition or the writer, is
 * launched in plain stream order, with no overlap. The decode, gather and prefill write
 * none of these inputs. For kernels of other code the caller keeps the rules (an event
 * wait or a call of this library in between also ends the overlap).
 * enable = 0 (default): ordinary stream order. Returns EKV_ERR_INVALID_ARG for a
 * null context or another value. */
ekv_status ekv_set_pdl(ekv_ctx* ctx, int enable);

/* Number of SMs and split-K CTAs per decode launch the context uses. */
ekv_status ekv_query(ekv_ctx* ctx, int* num_sms, int* split_ctas);

/* Static string for a status code. */
const char* ekv_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* EKV_H */
