/*
 * qa.h -- paged GQA attention for Qwen3-ASR-shaped serving, C ABI.
 *
 * Plain C99, extern "C".  The shared library libqa.so exports only the qa_*
 * symbols declared here; every kernel and helper stays hidden.  The
 * conventions follow the qwenasr.cpp public ABI (qwenasr.cpp ARCHITECTURE.md,
 * "Public API" and "ABI guarantee"): integer status codes with the same
 * numbering, a thread-local last-error message, a version string, and an
 * abi_version field that callers set through the default-params helper and
 * that the entry points check against the closed range
 * [QA_ABI_MIN_VERSION, QA_ABI_VERSION].
 *
 * Three operations make up the attention core:
 *
 *   qa_decode_attn   batched single-token decode over a paged KV cache with
 *                    grouped-query attention (16 query heads over 8 KV heads,
 *                    head_dim 128).  qwenasr.cpp ARCHITECTURE.md, "Qwen3
 *                    Thinker decoder" (decode appends one position at cur_len
 *                    and attends over [0, cur_len + 1)) and "GGUF layout"
 *                    (head_count 16, head_count_kv 8, key_length 128); M*
 *                    "Speech recognition: Whisper and Qwen3-ASR", "Graph"
 *                    (decode runs on paged KV) and "Serving notes" (pages).
 *   qa_prefill_attn  ragged causal prefill of packed prompts, writing the
 *                    fresh K/V into their pages.  qwenasr.cpp ARCHITECTURE.md,
 *                    "Qwen3 Thinker decoder" (prefill rewinds the cache, writes
 *                    K/V at [n_past, n_past + T) and attends over
 *                    [0, n_past + T)); M* page, "Graph" (prefill on packed
 *                    token buckets).
 *   qa_window_attn   bidirectional attention confined to windows of the
 *                    packed encoder sequence.  qwenasr.cpp ARCHITECTURE.md,
 *                    "Windowed audio tower" (block-diagonal mask over windows
 *                    of 104 tokens, plain bidirectional MHA, 1/sqrt(head_dim));
 *                    M* page, "Graph" (one packed forward with one segment per
 *                    window of every request).
 *
 * Common rules
 *
 *   - Every tensor argument is a DEVICE pointer to caller-owned memory,
 *     row-major and contiguous, except where a function says "host".  The
 *     library allocates nothing during a call.
 *   - bf16 means IEEE bfloat16.  Inputs are bf16; scores and softmax run in
 *     fp32; outputs are rounded to bf16 (round to nearest even).  (OneSpeech
 *     Qwen3 page, "Front end and graph numerics": score and softmax
 *     intermediates in float32, attended output rounded to bfloat16.)
 *   - Calls are asynchronous on params->stream (NULL = the legacy default
 *     stream) unless params->debug_checks is set, in which case the call
 *     synchronises the stream and reports device-side errors.
 *   - Host-checkable errors (NULL pointers, unsupported shapes, a workspace
 *     that is too small, a bad abi_version) return QA_STATUS_INVALID_PARAMS
 *     before anything is launched and set qa_last_error().  A failed launch
 *     returns QA_STATUS_LAUNCH_FAILED.
 *   - Device-side checks never fault or trap: a page id outside
 *     [0, num_pages), a sequence longer than its page-table row, a malformed
 *     cu_* array or an expired bounded wait skips the affected work and sets
 *     a bit in a per-library device status word, which qa_device_status()
 *     (or a debug_checks call) reads and clears.
 *   - Decode layout of the paged pool: [num_pages][page_size][n_kv_heads]
 *     [head_dim], token-major inside a page like the packed [T][Hkv][D] rows.
 *     Query head h reads KV head h / (n_q_heads / n_kv_heads) (contiguous
 *     GQA grouping).
 */
#ifndef QA_H
#define QA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QA_ABI_VERSION 2
#define QA_ABI_MIN_VERSION 1

/* Status codes: numbering of the qwenasr.cpp public ABI ("Public API");
 * -2 (load failed) and -5 (cancelled) have no use here.  -6 is new: a kernel
 * reported an error through the device status word. */
typedef enum qa_status {
    QA_STATUS_OK = 0,
    QA_STATUS_INVALID_PARAMS = -1,
    QA_STATUS_LAUNCH_FAILED = -3,
    QA_STATUS_OOM = -4,
    QA_STATUS_DEVICE_ERROR = -6
} qa_status;

/* Bits of the device status word (qa_device_status). */
#define QA_DEVICE_BAD_PAGE 0x1u     /* page id outside [0, num_pages)            */
#define QA_DEVICE_BAD_LENGTH 0x2u   /* seq_len < 0 or > max_pages * page_size    */
#define QA_DEVICE_BAD_SEGMENTS 0x4u /* cu_seqlens / cu_windows not monotonic, or
                                       not ending at total_tokens               */
#define QA_DEVICE_TIMEOUT 0x8u      /* a bounded wait inside a kernel expired    */

typedef struct qa_attn_params {
    int abi_version;       /* set by qa_attn_default_params()                    */
    int n_q_heads;         /* decode/prefill: 16; window: 14                     */
    int n_kv_heads;        /* decode/prefill: 8;  window: must equal n_q_heads   */
    int head_dim;          /* decode/prefill: 128; window: 64 or 128             */
    int page_size;         /* tokens per page; 16                                */
    int num_pages;         /* pool size P (pages in k_pages and v_pages)         */
    int max_pages_per_seq; /* page_table row stride                              */
    float scale;           /* softmax scale; 0 => 1/sqrt(head_dim)               */
    void *stream;          /* cudaStream_t; NULL => legacy default stream        */
    void *workspace;       /* decode scratch (device), caller-owned              */
    size_t workspace_bytes;
    int debug_checks;      /* 1 => synchronise and report device-side errors     */
    int stable_metadata;   /* ABI 2: 0, 1 or 2 (below); ignored if abi_version < 2 */
} qa_attn_params;

/* stable_metadata (decode calls: qa_decode_attn, qa_decode_attn_noalloc,
 * qa_decode_step; prefill calls: see after this paragraph).  The decode
 * kernel is launched as a programmatic dependent
 * of the kernel before it on the stream, so its CTAs may start while that
 * kernel is still finishing.  With stable_metadata = 1 the caller promises
 * that seq_lens and page_table are not written by any kernel that may still
 * be running when this call's kernel starts: the kernel directly before it on
 * the stream, and, if that one lets its successor start before it has waited
 * for its own predecessor, the kernels it waits for.  (Every kernel of this
 * library lets its successor start only after its own wait.)  A decode step
 * whose lengths and page table are copied in, or written by a kernel followed
 * by at least one other kernel, before its first layer meets this.  The
 * kernel then reads them, computes its work split and fetches its first page
 * ids before that kernel has finished, and waits only before it reads q, the
 * pools or the workspace or writes any output.  With 2 the caller promises the
 * same of k_pages and v_pages, and the kernel also streams its first pages
 * into shared memory before that wait.  Back-to-back layers of a decode step
 * (each reads its own layer's pools) and qa_decode_step (it writes the new
 * row itself) meet this; a decode after a qa_decode_append into the same
 * pools does not.  With 0 (the default) it waits before reading anything.
 * Other values are rejected.
 *
 * Prefill calls (qa_prefill_attn, qa_prefill_chunk_attn) launch the same
 * way.  With stable_metadata >= 1 the caller promises the same of cu_seqlens,
 * page_table and n_past; the kernel then maps its job, checks it, reads its
 * page ids and sets up its barriers and tensor memory before that wait, and
 * waits before it reads q, k, v or the pools or writes any output or page.
 * (1 and 2 act alike for prefill.) */

/* Defaults: abi_version = QA_ABI_VERSION, 16/8/128 heads, page_size 16,
 * scale 0 (1/sqrt(head_dim)), stream NULL, no workspace, debug_checks 0,
 * stable_metadata 0.
 * num_pages and max_pages_per_seq are 0 and must be set by the caller. */
qa_attn_params qa_attn_default_params(void);

/* Bytes of device workspace qa_decode_attn needs for `batch` requests on the
 * CURRENT device with these params: the split-K partial results (one fp32
 * (max, sum, accumulator[head_dim]) record per query head per work segment)
 * and one int32 arrival counter per request.  The workspace must be
 * zero-filled once before its first use (e.g. cudaMemset); every call leaves
 * the counters at zero again, so it can be reused without clearing.
 * max_seq_len is the longest sequence the caller will pass (used only for
 * validation).  Returns 0 on invalid arguments and sets qa_last_error(). */
size_t qa_decode_workspace_size(int batch, int max_seq_len, const qa_attn_params *params);

/* Paged GQA decode: one query token per request.
 *
 *   q          bf16 [batch][n_q_heads][head_dim]
 *   k_pages    bf16 [num_pages][page_size][n_kv_heads][head_dim]
 *   v_pages    bf16, same layout as k_pages
 *   page_table int32 [batch][max_pages_per_seq]; entry j of row b is the
 *              physical page holding positions [j*page_size, (j+1)*page_size)
 *              of request b; entries past ceil(seq_lens[b]/page_size) are
 *              never read
 *   seq_lens   int32 [batch]: number of cached positions request b attends
 *              over, including the current token, whose K/V must already be
 *              in its page; 0 gives a zero output row
 *   out        bf16 [batch][n_q_heads][head_dim]
 *
 * out[b][h] = softmax_j(q[b][h] . K_b[j] * scale) . V_b[j] over
 * j in [0, seq_lens[b]).  Slots past seq_lens[b] in the last page are never
 * read into the result (they may hold anything, NaN included).
 * Supported: head_dim 128, page_size 16, n_kv_heads in [1, 8],
 * n_q_heads / n_kv_heads in {1, 2}.  Needs params->workspace of at least
 * qa_decode_workspace_size(batch, ...) bytes, 256-byte aligned, zero-filled
 * before its first use (see qa_decode_workspace_size).  Calls sharing one
 * workspace must be ordered (one stream), since they share its counters.
 * q, page_table, seq_lens and out are read and written with plain loads and
 * stores (only the pools go through the bulk-copy engine), so they may also
 * be page-locked host memory that the device addresses directly (cudaHostAlloc
 * under unified addressing): a serving step then needs no copies of its own,
 * the kernel moves those bytes over the host link itself. */
qa_status qa_decode_attn(const void *q, const void *k_pages, const void *v_pages,
                         const int32_t *page_table, const int32_t *seq_lens, int batch,
                         void *out, const qa_attn_params *params);

/* Paged GQA decode for callers that cannot allocate device memory.
 *
 * Not part of the method described by the Qwen3-ASR pages (they have no
 * counterpart): a convenience for callers that cannot call cudaMalloc -- for
 * example a plugin whose host application owns every device allocation, a
 * real-time path that may not wait on or fail in an allocator, or plain C
 * code without an allocator of its own.  Same arguments, layouts and result
 * as qa_decode_attn, but params->workspace is ignored: the split-K scratch
 * lives in a fixed 4 MiB array inside the library, reserved on every GPU that
 * loads it until the process exits.  Nothing is allocated.
 *
 *   - A batch whose scratch would exceed 4 MiB is rejected with
 *     QA_STATUS_INVALID_PARAMS and a message giving the sizes (with 16 query
 *     heads and head_dim 128 about 330 requests fit on a 152-SM GPU).
 *   - All calls on a device share the array: calls whose kernels overlap on
 *     the GPU (unordered streams or host threads) race and give wrong
 *     results.  Calls ordered on one stream are safe.  The array keeps the
 *     last call's contents; the only part that must start at zero (the
 *     per-request arrival counters) starts zeroed and every call leaves it
 *     zeroed, so nothing needs clearing between calls.
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress) and hands it to the kernel; nothing is cached,
 *     so a cudaDeviceReset between calls does not leave a stale address.
 *   - Argument checks are those of qa_decode_attn (stable_metadata included),
 *     except that there is no workspace to check. */
qa_status qa_decode_attn_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                 const int32_t *page_table, const int32_t *seq_lens, int batch,
                                 void *out, const qa_attn_params *params);

/* Ragged causal prefill with the KV page write.
 *
 *   q          bf16 [total_tokens][n_q_heads][head_dim], requests packed
 *   k, v       bf16 [total_tokens][n_kv_heads][head_dim]
 *   cu_seqlens int32 [batch + 1]: request r owns rows [cu[r], cu[r+1]);
 *              cu[0] = 0, cu[batch] = total_tokens, non-decreasing
 *   page_table int32 [batch][max_pages_per_seq]: destination pages
 *   k_pages, v_pages  destination pools (layout as in qa_decode_attn)
 *   out        bf16 [total_tokens][n_q_heads][head_dim]
 *
 * Writes row i of request r, bit for bit, to page page_table[r][i/page_size]
 * slot i % page_size of both pools (positions [0, len) of each request:
 * n_past = 0, the cache was rewound), and computes
 * out[t][h] = softmax over j <= t within the request of q[t][h] . k[j][g]
 * (g = h / group) times v[j][g], from the packed k and v.  Pool slots that no
 * row maps to are left untouched.  Rows are checked on the device: a page id
 * outside [0, num_pages) sets QA_DEVICE_BAD_PAGE and that row is not written;
 * a request longer than max_pages_per_seq * page_size sets
 * QA_DEVICE_BAD_LENGTH, and its rows past that bound are not written to the
 * pools (nor, past the next multiple of 128, attended: those out rows are left
 * as they were).
 * Supported: head_dim 128, page_size 16, n_q_heads / n_kv_heads in {1, 2}. */
qa_status qa_prefill_attn(const void *q, const void *k, const void *v,
                          const int32_t *cu_seqlens, int batch, int total_tokens,
                          const int32_t *page_table, void *k_pages, void *v_pages, void *out,
                          const qa_attn_params *params);

/* Chunked prefill: new prompt rows after n_past cached positions.
 *
 * qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder": a forward writes its
 * fresh K/V into the cache at [n_past, n_past + T) and attends over
 * [0, n_past + T) (causal, aligned at the end).  Request r already holds
 * n_past[r] positions in its pages (page_table row r); its new rows are
 * packed as in qa_prefill_attn.  New row i (position n_past[r] + i) attends
 * over every cached position [0, n_past[r]) (read through the page table)
 * and over the new rows j <= i (from the packed k, v); the new rows are
 * written bit for bit to positions n_past[r] + i.  With every n_past = 0
 * this is qa_prefill_attn.
 *
 *   n_past     int32 [batch] (device): cached positions per request
 *   other arguments as in qa_prefill_attn
 *
 * Device checks: n_past outside [0, max_pages_per_seq * page_size] or
 * n_past + new rows beyond it sets QA_DEVICE_BAD_LENGTH (the request is
 * skipped, or its rows past the page-table row are not written); a page id
 * outside [0, num_pages) among the cached or new positions sets
 * QA_DEVICE_BAD_PAGE.  Supported as qa_prefill_attn. */
qa_status qa_prefill_chunk_attn(const void *q, const void *k, const void *v,
                                const int32_t *cu_seqlens, const int32_t *n_past, int batch,
                                int total_tokens, const int32_t *page_table, void *k_pages,
                                void *v_pages, void *out, const qa_attn_params *params);

/* Decode KV append with per-head QK-norm and NEOX RoPE (one new token per
 * request), the step that precedes qa_decode_attn in a decode layer.
 *
 * qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder": per layer, q and k
 * get a per-head RMSNorm (RMS over head_dim, then a [head_dim] gain), then a
 * 1D NEOX RoPE (freq_base 1e6; "Attention and RoPE": rotate half); decode
 * appends the new token at position cur_len and attends over
 * [0, cur_len + 1).  With cur = seq_lens[b] - 1 and D = head_dim:
 *
 *   y[d] = x[d] / sqrt(mean_d x[d]^2 + rms_eps) * gain[d]
 *   a_i  = cur * rope_theta^(-2 i / D),                 i in [0, D/2)
 *   z[i] = y[i] cos a_i - y[i + D/2] sin a_i,  z[i + D/2] = y[i] sin a_i + y[i + D/2] cos a_i
 *
 *   q          bf16 [batch][n_q_heads][head_dim]   pre-norm query projection
 *   k, v       bf16 [batch][n_kv_heads][head_dim]  pre-norm key, value projections
 *   q_gain, k_gain  float [head_dim]               the two RMSNorm gains
 *   rms_eps    > 0 (1e-6 for the Qwen3 decoders); rope_theta > 0 (1e6)
 *   page_table, seq_lens  as in qa_decode_attn; seq_lens[b] >= 1 counts the
 *              new token
 *   k_pages, v_pages  pools [num_pages][page_size][n_kv_heads][head_dim]:
 *              slot cur % page_size of page page_table[b][cur / page_size]
 *              receives z of k (bf16) and v unchanged
 *   q_out      bf16 [batch][n_q_heads][head_dim]: z of q (bf16), the query
 *              for qa_decode_attn; may be q itself (in place), must not
 *              otherwise overlap an input
 *
 * Arithmetic in fp32.  Each angle is carried as an exact sum of fp32 terms
 * (frequencies computed on the host in fp64, passed as fp32 hi + lo parts)
 * and reduced modulo 2 pi by the Cody-Waite three-constant scheme before an
 * fp32 sin/cos; results rounded to bf16, nearest even.  One launch (one CTA per
 * request), asynchronous on params->stream, launched so that a following
 * qa_decode_attn on the same stream can start its launch early.  Device
 * checks: seq_lens[b] outside [1, max_pages_per_seq * page_size] sets
 * QA_DEVICE_BAD_LENGTH and a page id outside [0, num_pages) sets
 * QA_DEVICE_BAD_PAGE; such a request is skipped entirely (q_out row
 * unwritten).  params->scale is not used.
 * Supported: head_dim 128, page_size 16, n_q_heads / n_kv_heads in {1, 2},
 * max_pages_per_seq * page_size <= 262144 (positions below 2^18). */
qa_status qa_decode_append(const void *q, const void *k, const void *v, const float *q_gain,
                           const float *k_gain, float rms_eps, float rope_theta,
                           const int32_t *page_table, const int32_t *seq_lens, int batch,
                           void *k_pages, void *v_pages, void *q_out, const qa_attn_params *params);

/* The fused decode step: qa_decode_append and qa_decode_attn in one launch.
 *
 * Same arguments and results as calling qa_decode_append (q, k, v, gains,
 * rms_eps, rope_theta, pools, page_table, seq_lens) and then qa_decode_attn
 * on its rotated query (workspace, scale and out as in qa_decode_attn), but
 * the rotated query never leaves the chip: every CTA normalises and rotates
 * the query heads it reads, and the CTA that holds a request's last page
 * normalises and rotates the new key, writes the new K/V row to its slot and
 * uses it from shared memory in place of the slot's old contents.  No grid
 * waits on another.  The rotated query is rounded to bf16 before use, as in
 * the two-call sequence; results agree with it up to fp32 evaluation order.
 * Device checks as in both calls (a request with seq_lens[b] = 0 sets
 * QA_DEVICE_BAD_LENGTH here, since it has no new token).
 * Supported: as qa_decode_append; k, v and the gains 16-byte aligned. */
qa_status qa_decode_step(const void *q, const void *k, const void *v, const float *q_gain,
                         const float *k_gain, float rms_eps, float rope_theta, void *k_pages,
                         void *v_pages, const int32_t *page_table, const int32_t *seq_lens,
                         int batch, void *out, const qa_attn_params *params);

/* Captured steps (CUDA graphs): a decode step of n_layers qa_decode_attn
 * calls, or a prefill step of a packed bucket of n_layers qa_prefill_attn
 * calls, captured once and replayed with one launch.  M* "Speech recognition:
 * Whisper and Qwen3-ASR", "Serving notes": steps are captured per decode batch
 * size and per packed prefill bucket and replayed.
 *
 *   q, k, v, k_pages, v_pages, out: arrays of n_layers device pointers, layer
 *   i's tensors as for the single call; page_table, seq_lens / cu_seqlens,
 *   batch, total_tokens and params (including the decode workspace, shared by
 *   the layers, which run one after another) are common to all layers.
 *
 * Every pointer and size is fixed at capture.  A replay (qa_graph_launch on
 * any stream of the capturing device) reads the buffers' contents at replay
 * time: refill q, lengths, page table and so on in place between replays;
 * for another batch size or bucket, capture another graph.  The capture
 * validates each call exactly as the single call does (returning its status
 * and message); params->debug_checks must be 0 (it synchronises).  The pointer
 * arrays themselves are read during the call only.  Make one ordinary call of
 * each operation on the device before the first capture (it loads the
 * kernels).  qa_graph_destroy releases the graph (NULL is ignored). */
typedef struct qa_graph qa_graph;
qa_status qa_decode_graph_create(int n_layers, const void *const *q, const void *const *k_pages,
                                 const void *const *v_pages, const int32_t *page_table,
                                 const int32_t *seq_lens, int batch, void *const *out,
                                 const qa_attn_params *params, qa_graph **graph);
qa_status qa_prefill_graph_create(int n_layers, const void *const *q, const void *const *k,
                                  const void *const *v, const int32_t *cu_seqlens, int batch,
                                  int total_tokens, const int32_t *page_table, void *const *k_pages,
                                  void *const *v_pages, void *const *out, const qa_attn_params *params,
                                  qa_graph **graph);
qa_status qa_graph_launch(qa_graph *graph, void *stream);
void qa_graph_destroy(qa_graph *graph);

/* Windowed bidirectional attention over a packed sequence.
 *
 *   q, k, v    bf16 [total_tokens][n_q_heads][head_dim] (n_kv_heads must equal
 *              n_q_heads: plain MHA)
 *   cu_windows int32 [n_windows + 1]: window w owns rows
 *              [cu_windows[w], cu_windows[w+1]); cu_windows[0] = 0,
 *              cu_windows[n_windows] = total_tokens, non-decreasing
 *   out        bf16 [total_tokens][n_q_heads][head_dim]
 *
 * Every row attends over all rows of its own window and nothing else.
 * Supported: head_dim 64 or 128, windows of any length.
 *
 * params->workspace is optional.  Without one, the (window, head) jobs go to
 * the persistent grid's CTAs in a fixed order.  With one (at least
 * qa_window_workspace_size() bytes, 4-byte aligned, zero-filled before its
 * first use), CTAs claim the jobs one at a time from a counter in it, so
 * CTAs that start later or run slower take fewer jobs; each call leaves the
 * counter zero again.  Calls sharing one workspace must be ordered (one
 * stream).  The result is the same bit for bit either way. */
qa_status qa_window_attn(const void *q, const void *k, const void *v,
                         const int32_t *cu_windows, int n_windows, int total_tokens, void *out,
                         const qa_attn_params *params);

/* Bytes of the optional qa_window_attn workspace (its job counter). */
size_t qa_window_workspace_size(void);

/* Window plan (HOST helper, host pointers).  Cuts each request's encoder
 * tokens into consecutive windows of window_tokens tokens counted from the
 * request's own start, the last window partial (qwenasr.cpp ARCHITECTURE.md,
 * "Windowed audio tower": windows of window_aftercnn = conv_out(chunk_mel) *
 * window_chunks = 13 * 8 = 104 tokens).  A request with no token gives no
 * window.  window_tokens <= 0 selects 104.
 *
 *   token_counts  host int32 [n_requests]
 *   cu_windows    host int32 [capacity]; receives n_windows + 1 offsets
 *
 * Returns the number of windows, or -1 (and sets qa_last_error()) on a
 * negative count, a capacity that is too small, or int32 overflow. */
int qa_window_plan(const int32_t *token_counts, int n_requests, int window_tokens,
                   int32_t *cu_windows, int capacity);

/* ------------------------------------------------------------------------
 * The AuT encoder layer around the window attention (qwenasr.cpp
 * ARCHITECTURE.md, "Windowed audio tower": pre-norm Whisper-style layer,
 * LayerNorm with bias, bias on q / k / v / output, gelu MLP; "GGUF layout":
 * attn_norm, attn_q / attn_k / attn_v / attn_output, ffn_norm, ffn_up /
 * ffn_down, each with weight and bias).  All tensors are caller-owned bf16
 * device buffers; every row stride is the row's own width.  Linear weights
 * keep the PyTorch (out, in) layout ("Tensor shape and layout"): y = x W^T.
 * ------------------------------------------------------------------------ */

/* Weights of one layer (device pointers, bf16). */
typedef struct qa_encoder_weights {
    const void *ln1_g, *ln1_b;  /* [d_model] attention LayerNorm gain, bias   */
    const void *w_qkv, *b_qkv;  /* [3 d_model][d_model], [3 d_model]: the q,  */
                                /* k and v projections stacked in that order */
    const void *w_o, *b_o;      /* [d_model][d_model], [d_model]              */
    const void *ln2_g, *ln2_b;  /* [d_model] MLP LayerNorm gain, bias         */
    const void *w_fc1, *b_fc1;  /* [d_ffn][d_model], [d_ffn]                  */
    const void *w_fc2, *b_fc2;  /* [d_model][d_ffn], [d_model]                */
} qa_encoder_weights;

/* Workspace bytes (256-byte aligned start) that qa_encoder_layer needs for
 * total_tokens tokens: the layer's bf16 intermediates (LayerNorm output,
 * q|k|v, attention output, residual stream h, MLP hidden).  0 on bad sizes. */
size_t qa_encoder_workspace_size(int total_tokens, int d_model, int d_ffn);

/* One encoder layer over total_tokens packed tokens cut into windows:
 *
 *   a = LN1(x);  q|k|v = a Wqkv^T + bqkv;  o = window attention(q, k, v)
 *   h = x + (o Wo^T + bo);  f = gelu(LN2(h) W1^T + b1)
 *   out = h + (f W2^T + b2)
 *
 * LN(v) = (v - mean) / sqrt(var + ln_eps) * g + b over each row (biased
 * variance); gelu the exact u / 2 (1 + erf(u / sqrt 2)); the attention is
 * qa_window_attn's (n_heads heads of d_model / n_heads dims, scale
 * 1 / sqrt(head_dim)).  Each line's result is rounded to bf16; inside a line
 * accumulation is fp32.
 *
 *   x, out     bf16 [total_tokens][d_model] (may not alias)
 *   cu_windows int32 [n_windows + 1], as for qa_window_attn
 *   params     stream, debug_checks, and workspace / workspace_bytes of at
 *              least qa_encoder_workspace_size(); the head fields are unused
 *
 * Supported: d_model a multiple of 128 up to 2048 with d_model / n_heads 64
 * or 128, d_ffn a multiple of 8.  Seven kernel launches, asynchronous on the
 * stream. */
qa_status qa_encoder_layer(const void *x, const int32_t *cu_windows, int n_windows, int total_tokens,
                           int d_model, int n_heads, int d_ffn, const qa_encoder_weights *weights,
                           float ln_eps, void *out, const qa_attn_params *params);

/* One projection of the layer on the tensor cores:
 *
 *   out[i][j] = act(sum_k x[i][k] w[j][k] + bias[j]) + residual[i][j]
 *
 *   x [m][k], w [n][k], bias [n] or NULL, residual [m][n] or NULL, out
 *   [m][n]: bf16, row-major, rows packed; act 0 (none) or 1 (exact gelu).
 * fp32 accumulation, bf16 result.  Supported: k and n multiples of 8.  Only
 * params->stream and debug_checks are used. */
qa_status qa_linear(const void *x, int m, int k, const void *w, int n, const void *bias, int act,
                    const void *residual, void *out, const qa_attn_params *params);

/* LayerNorm over each row of x [t][d] with gain and bias [d] (bf16), result
 * bf16 [t][d] (may alias x).  Supported: d a multiple of 128 up to 2048.
 * Only params->stream and debug_checks are used. */
qa_status qa_layer_norm(const void *x, int t, int d, const void *gain, const void *bias, float eps, void *y,
                        const qa_attn_params *params);

/* Synchronises `stream` (cudaStream_t, NULL = legacy default), then reads and
 * clears the device status word of the current device.  Returns its bits
 * (QA_DEVICE_*), 0 when nothing went wrong, or -1 on a CUDA error. */
int qa_device_status(void *stream);

/* Exercises the failure path of the kernels' waits without a fault: launches
 * one CTA (asynchronous on `stream`) that waits, through the same bounded
 * wait the attention kernels use, on a barrier that nothing ever completes.
 * The wait gives up after limit_us microseconds (1 .. 1000000; the kernels
 * themselves give up after 2 s), sets QA_DEVICE_TIMEOUT in the device status
 * word and the kernel ends; the context stays usable.  Read the bit with
 * qa_device_status().  INVALID_PARAMS for a limit outside that range,
 * LAUNCH_FAILED on a launch error. */
qa_status qa_check_bounded_wait(unsigned int limit_us, void *stream);

/* Thread-local message describing the last failure on this thread; valid
 * until the next qa_* call on the same thread.  Never NULL. */
const char *qa_last_error(void);

/* Library version string ("qa-attn <version> abi <n>"). */
const char *qa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QA_H */
