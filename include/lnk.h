/*
 * lnk.h -- C ABI of liblnk: paged decode / step attention for GB300 (sm_103a).
 *
 * One layer's attention step of a paged decoder-serving engine:
 *
 *   lnk_paged_append_rope   rotate the step's q/k with RoPE (after an optional
 *                           per-head QK-norm) and write each token's k/v into
 *                           its slot of the shared page pool;
 *   lnk_paged_decode_attn   one query token per decode row over that row's pages
 *                           (the serving step "decode_paged");
 *   lnk_paged_decode_step   append_rope then decode_attn for one token per
 *                           decode row (one kernel for small launches);
 *   lnk_paged_step_attn     packed prompt chunks plus decode rows in one call
 *                           ("step_paged"; with no decode rows it is
 *                           "prefill_paged").
 *
 * Sources: the model pages "Mistral 7B Instruct v0.3", "Qwen3-4B" and
 * "Llama 3.1 8B Instruct", Entries table (prefill_paged, decode_paged,
 * step_paged); "Phi-3 Mini 4K Instruct -- files", src/attention.linnet
 * (decode_rows, prefill_packed, step_packed, window_mask) and src/rope.linnet
 * (tables); "Llama 3.1 8B Instruct", rope-scaling paragraph; "Qwen3-4B",
 * QK-norm paragraph.
 *
 * Conventions (all entry points)
 *   - bf16 tensors are IEEE bfloat16 bit patterns (lnk_bf16), row-major and
 *     contiguous in the stated shape.  int32 arrays are contiguous.
 *   - Every pointer argument named "device" is device memory owned by the
 *     caller; the library allocates nothing, frees nothing and never
 *     synchronises.  Work is enqueued on `stream` (NULL = legacy default).
 *   - Pool layout: k_pool and v_pool are [num_kv_heads][num_pages * 64][head_dim]
 *     bf16 (the caches' [Batch = 1, KvHeads, MaxSeq, D] with MaxSeq =
 *     num_pages * 64).  Logical position j of table row r lives in pool slot
 *     table[r * pages_per_row + j / 64] * 64 + j % 64.  Pool pointers must be
 *     16-byte aligned.
 *   - Host-detectable argument errors return a status synchronously and
 *     enqueue nothing.  Data-dependent errors found on the device (a table
 *     entry outside [0, num_pages), a position past the table row, a bad row
 *     or slot) make the affected token or page skip its work and OR a
 *     LNK_DEV_* bit into *dev_status (an int32 in device memory; NULL = do
 *     not report).  No kernel traps or faults on bad data.
 *   - A negative position marks an inactive token or row: nothing is written
 *     for it and its outputs are zero.  This is not an error.
 *   - Ordering: attention reads the slots append_rope writes, so call
 *     append_rope first on the same stream.
 */
#ifndef LNK_H
#define LNK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lnk_bf16;          /* bfloat16 bit pattern */
typedef struct CUstream_st* lnk_stream; /* same type as cudaStream_t */

typedef enum lnk_status {
  LNK_OK = 0,
  LNK_EINVAL = 1,          /* null pointer, misaligned pointer, inconsistent shape */
  LNK_ERANGE = 2,          /* a size outside the supported range */
  LNK_ECUDA = 3,           /* a CUDA runtime call failed (launch, attribute, ...) */
  LNK_EUNSUPPORTED = 4,    /* head_dim, group size or page size not supported */
  LNK_EWORKSPACE = 5,      /* workspace NULL or smaller than lnk_paged_workspace_size */
  LNK_ENOSPACE = 6         /* the page allocator has too few free pages (or host memory ran out) */
} lnk_status;

/* Bits ORed into *dev_status by the kernels. */
#define LNK_DEV_BAD_ROW      0x01  /* a token's row outside [0, num_rows) */
#define LNK_DEV_BAD_POSITION 0x02  /* position >= pages_per_row * 64 */
#define LNK_DEV_BAD_PAGE     0x04  /* a table entry outside [0, num_pages) on a read or write path */
#define LNK_DEV_BAD_SLOT     0x08  /* slots[t] outside [0, num_pages * 64) */
#define LNK_DEV_SEGMENT      0x10  /* adjacent chunk tokens share a segment but not a row */
#define LNK_DEV_BAD_LAST     0x20  /* last[m] outside [0, P) */
#define LNK_DEV_TIMEOUT      0x40  /* a pipeline wait gave up (never expected) */

/* Shape of one attention layer and its page pool. */
typedef struct lnk_attn_desc {
  int32_t num_q_heads;    /* Hq */
  int32_t num_kv_heads;   /* Hkv; Hq % Hkv == 0 and Hq / Hkv in {1, 2, 4, 8} */
  int32_t head_dim;       /* D in {64, 96, 128} */
  int32_t page_size;      /* positions per page; must be 64 */
  int32_t num_pages;      /* pages in each of k_pool / v_pool */
  int32_t num_rows;       /* rows of table */
  int32_t pages_per_row;  /* columns of table (its row stride, in entries) */
  int32_t window;         /* 0: none; else key j is visible to a query at p
                             iff p - window < j <= p (itself and window - 1 before) */
  float scale;            /* softmax scale; 0 selects 1 / sqrt(head_dim) */
  int32_t kv_dtype;       /* element type of k_pool / v_pool: LNK_KV_BF16 (0, the
                             pages' pools) or LNK_KV_E4M3 (8-bit pools, below) */
  float k_scale;          /* LNK_KV_E4M3: a K code c stands for e4m3(c) * k_scale (> 0, finite) */
  float v_scale;          /* LNK_KV_E4M3: a V code c stands for e4m3(c) * v_scale (> 0, finite) */
} lnk_attn_desc;

/* Pool element types (lnk_attn_desc.kv_dtype).
 *
 * LNK_KV_BF16: bfloat16 pools, as on the pages.
 * LNK_KV_E4M3: 8-bit pools (not on the pages; an option of this library that
 *   halves the bytes of the HBM-bound decode path).  Elements are OCP E4M3
 *   codes (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
 *   subnormals, no infinities, S.1111.111 = NaN, largest finite 448), one
 *   byte each: the pools are [Hkv][num_pages * 64][D] bytes and the lnk_bf16*
 *   pool arguments of every entry point point to those bytes.  The append
 *   stores code = round-to-nearest-even E4M3 of fl32(value / scale), where
 *   value is the bf16 value a bf16 pool would hold (the rotated K, the V
 *   input) and the division is one IEEE float32 division, saturating to
 *   +-448.  Attention uses the dequantized values e4m3(c) * scale.  Chunk
 *   attention (P > 0 in lnk_paged_step_attn) is supported on bf16 pools only;
 *   decode rows are supported on both.  Decode over 8-bit pools converts the
 *   rotated queries to f16 (exactly, for magnitudes in [2^-14, 65504]): a
 *   query element above 65504 in magnitude becomes infinite there, and one
 *   below 2^-14 loses precision or becomes zero, so the queries must stay
 *   within that range (unit-scale projections do by far). */
#define LNK_KV_BF16 0
#define LNK_KV_E4M3 1

/* Rotary frequencies: inv_freq[i] = exp(-(f32(i) * 2 / f32(D)) * log(theta))
 * in float32 ("Phi-3 Mini 4K Instruct -- files", src/rope.linnet, tables),
 * optionally rescaled by wavelength in three bands ("Llama 3.1 8B Instruct",
 * rope-scaling paragraph): wavelen > orig / low_freq_factor -> inv / factor;
 * wavelen < orig / high_freq_factor -> inv; else linear blend with
 * smooth = (orig / wavelen - low) / (high - low). */
typedef struct lnk_rope_desc {
  double theta;                   /* rotary base (as float32, like the pages) */
  int32_t llama3;                 /* 0: plain; 1: llama3 three-band rescale */
  double factor;                  /* llama3: 8 for Llama 3.1 */
  double low_freq_factor;         /* llama3: 1 */
  double high_freq_factor;        /* llama3: 4 */
  double original_max_position;   /* llama3: 8192 */
} lnk_rope_desc;

/* Human-readable name of a status. */
const char* lnk_status_string(lnk_status status);

/* Host-only: the float32 frequency table the append kernel uses, written to
 * out[0 .. head_dim/2).  Same definition as lnk_rope_desc's comment; log and
 * exp are taken correctly rounded, the llama3 rescale in double rounded once. */
lnk_status lnk_rope_inv_freq(const lnk_rope_desc* rope, int32_t head_dim, float* out);

/* Bytes of device workspace that decode_attn / step_attn need for up to
 * max_rows decode rows on the current device.  Returns 0 on bad arguments.
 * The workspace must be zero-filled once before its first use (it holds
 * counters that every completed call leaves at zero); zero it again only after
 * a call reported LNK_DEV_TIMEOUT.  Calls that share a workspace must not run
 * concurrently. */
size_t lnk_paged_workspace_size(const lnk_attn_desc* desc, int32_t max_rows);

/*
 * lnk_paged_append_rope -- per token: optional QK-norm, RoPE, K/V append.
 *
 * Defines: "Qwen3-4B" QK-norm paragraph (RMS over each head's head_dim slice,
 * eps, weight gamma, after the head split, before rope); "Phi-3 Mini 4K
 * Instruct -- files" src/rope.linnet tables (angle f32(position) * inv_freq[i],
 * each frequency used for both halves: element i turns with element i + D/2)
 * and src/attention.linnet write_tokens; "Mistral 7B Instruct v0.3" Entries
 * table, prefill_paged ("each token written at its place in the pool").
 *
 *   q        device [T][Hq][D]   projected queries
 *   k, v     device [T][Hkv][D]  projected keys / values
 *   positions device int32 [T]   position of each token in its row (< 0: inactive)
 *   rows     device int32 [T]    table row of each token; NULL: token t uses row t
 *   slots    device int32 [T]    pool slot to write; NULL: derived from the table
 *   table    device int32 [num_rows][pages_per_row] (unused when slots != NULL)
 *   q_norm_w, k_norm_w  device [D] QK-norm weights, or NULL for no QK-norm
 *   norm_eps QK-norm epsilon (1e-6 for Qwen3)
 *   k_pool, v_pool  device pools (written at the tokens' slots only; 8-bit
 *            codes for LNK_KV_E4M3, see lnk_attn_desc.kv_dtype)
 *   q_out    device [T][Hq][D]   rotated queries (zero for inactive tokens)
 *   T        tokens (0 is allowed and enqueues nothing)
 *
 * Numerics: QK-norm, cos/sin of the float32 angle and the rotation are
 * evaluated to about 2^-46 relative (float pairs; double precision for
 * angles of 2^20 and more and for the QK-norm factor) and rounded once to
 * bf16 (nearest even); v is copied bit for bit.  Two tokens writing one slot
 * race (the engine's padding tokens write a shared dump slot nobody reads).
 *
 * Ordering with the preceding kernel: the append kernel is launched as a
 * programmatic dependent launch and reads `positions`, `rows`, `slots` and
 * `table` (and only those) before it waits for the kernel before it on the
 * stream; q, k, v, the QK-norm weights, the pools and q_out are touched after
 * the wait.  So those four must not be written by the kernel immediately
 * preceding this call on the same stream (this library's kernels only read
 * them).
 */
lnk_status lnk_paged_append_rope(const lnk_attn_desc* desc, const lnk_rope_desc* rope,
                                 const lnk_bf16* q, const lnk_bf16* k, const lnk_bf16* v,
                                 const int32_t* positions, const int32_t* rows,
                                 const int32_t* slots, const int32_t* table,
                                 const lnk_bf16* q_norm_w, const lnk_bf16* k_norm_w,
                                 float norm_eps, lnk_bf16* k_pool, lnk_bf16* v_pool,
                                 lnk_bf16* q_out, int32_t T, int32_t* dev_status,
                                 lnk_stream stream);

/*
 * lnk_paged_decode_attn -- one query token per decode row over its pages.
 *
 * Defines: "Mistral 7B Instruct v0.3" Entries table, decode_paged ("decode_rows
 * for serving from pages"); "Phi-3 Mini 4K Instruct -- files",
 * src/attention.linnet decode_rows (row b attends over itself up to
 * positions[b], with the window mask) and the scale rsqrt(head_dim).
 * Query head h reads kv head h / (Hq / Hkv).
 *
 *   q_roped  device [B][Hq][D]  rotated queries (q_out of append_rope), 16-byte aligned
 *   positions device int32 [B]  position of row b's token (< 0: inactive row)
 *   table    device int32 [num_rows][pages_per_row]; decode row b uses table row b
 *   k_pool, v_pool device pools (bf16, or 8-bit codes for LNK_KV_E4M3)
 *   out      device [B][Hq][D]  attention output (bf16, nearest even), 8-byte aligned
 *   B        decode rows, 0 <= B <= min(num_rows, 4096)
 *   workspace device scratch of ws_bytes >= lnk_paged_workspace_size(desc, B)
 *             (256-byte aligned; zero-filled before its first use, and again
 *             after a call that reported LNK_DEV_TIMEOUT; the kernel leaves
 *             its counters at zero otherwise)
 *
 * Ordering with the preceding kernel: the decode kernel is launched as a
 * programmatic dependent launch and reads `positions` and `table` (and only
 * those) before it waits for the kernel before it on the stream; q, the pools
 * and the workspace are touched after the wait.  (When every (row, kv head)
 * pair is one CTA's whole work, the kernel also asks L2 to prefetch the pair's
 * pool pages before the wait: a prefetch reads no values into the kernel, and
 * what the preceding kernel writes to those pages is what the kernel's copies
 * read after the wait.)  So `positions` and `table`
 * must not be written by the kernel immediately preceding this call on the
 * same stream (lnk_paged_append_rope only reads them); a caller that computes
 * them on the device should write them earlier, or put another operation in
 * between.  The decode kernel in turn lets the next kernel on the stream start
 * early (programmatic dependent launch): a kernel launched that way must wait
 * for it (griddepcontrol.wait) before reading `out` or writing what it reads.
 */
lnk_status lnk_paged_decode_attn(const lnk_attn_desc* desc, const lnk_bf16* q_roped,
                                 const int32_t* positions, const int32_t* table,
                                 const lnk_bf16* k_pool, const lnk_bf16* v_pool,
                                 lnk_bf16* out, int32_t B, void* workspace, size_t ws_bytes,
                                 int32_t* dev_status, lnk_stream stream);

/*
 * lnk_paged_decode_step -- a whole decode step: append, then attention.
 *
 * Defines: "Phi-3 Mini 4K Instruct -- files", src/attention.linnet
 * (decode_rows: write the row's new token at its position, then attend over
 * the row up to it); "Mistral 7B Instruct v0.3", Entries table (decode_paged).
 *
 * The same results as lnk_paged_append_rope(desc, rope, q, k, v, positions,
 * rows = NULL, slots = NULL, table, q_norm_w, k_norm_w, norm_eps, k_pool,
 * v_pool, q_out, T = B, ...) followed by lnk_paged_decode_attn(desc, q_out,
 * positions, table, k_pool, v_pool, out, B, ...), bit for bit: decode row b's
 * token is token b, written through table row b.  Arguments are those two
 * calls' (q_out must be 16-byte aligned); every check of both is made before
 * anything is enqueued.
 *
 * When B * num_kv_heads is at most the decode grid (one CTA per SM, two for
 * 8-bit pools when they fit) and at least half the SM count, and a (row, kv
 * head) pair can span at most 16 pages (pages_per_row, or the window's
 * pages), it is one kernel: the
 * CTA that attends for pair (b, h) first rotates that pair's query heads and
 * key head and writes its k/v row into the pool, then loads the row's pages
 * (the last one after that write).  Otherwise it is the two kernels above.
 * In the one-kernel form a token's pool slot must not be visible to another
 * decode row of the same call (rows share only pages below their positions,
 * as copy on write keeps them), and `positions` and `table` must not be
 * written by the kernel immediately preceding the call on the stream.
 */
lnk_status lnk_paged_decode_step(const lnk_attn_desc* desc, const lnk_rope_desc* rope,
                                 const lnk_bf16* q, const lnk_bf16* k, const lnk_bf16* v,
                                 const int32_t* positions, const int32_t* table,
                                 const lnk_bf16* q_norm_w, const lnk_bf16* k_norm_w,
                                 float norm_eps, lnk_bf16* k_pool, lnk_bf16* v_pool,
                                 lnk_bf16* q_out, lnk_bf16* out, int32_t B, void* workspace,
                                 size_t ws_bytes, int32_t* dev_status, lnk_stream stream);

/* Kernels that lnk_paged_decode_step enqueues for B rows on the current
 * device: 1 (the one-kernel form) or 2; 0 for B = 0; -1 for a descriptor or
 * B that the call would reject. */
int32_t lnk_paged_decode_step_launches(const lnk_attn_desc* desc, int32_t B);

/*
 * lnk_paged_step_attn -- packed prompt chunks and decode rows in one call.
 *
 * Defines: "Mistral 7B Instruct v0.3" Entries table, step_paged ("prefill_paged
 * and decode_paged in one pass") and prefill_paged (prompts packed end to end,
 * each token attending over its row's pages up to its position: chunks,
 * shared prefixes); "Phi-3 Mini 4K Instruct -- files", src/attention.linnet
 * step_packed / prefill_packed (prompt tokens first, then one token per row)
 * and src/lib.linnet prefill_packed (last[m] names prompt m's last token).
 *
 *   q_roped   device [P + B][Hq][D]: P chunk tokens, then B decode rows (16-byte aligned)
 *   rows      device int32 [P]  table row of each chunk token
 *   positions device int32 [P]  position of each chunk token (< 0: inactive)
 *   segments  device int32 [P]  prompt of each chunk token, or NULL.  Prompts
 *             live in their own rows, so a token sees only its own prompt (and
 *             that row's earlier context); adjacent tokens with equal segments
 *             must share a row (LNK_DEV_SEGMENT otherwise).
 *   step_positions device int32 [B]  decode row b's position; row b uses table row b
 *   table, k_pool, v_pool  as above
 *   out       device [P + B][Hq][D]
 *   last      device int32 [M] or NULL: chunk token whose output row is copied
 *             to last_out[m] (device [M][Hq][D]); M may be 0
 *   P, B      chunk tokens and decode rows (either may be 0); P > 0 with
 *             LNK_KV_E4M3 pools returns LNK_EUNSUPPORTED
 *   workspace as for decode_attn with max_rows >= B
 */
lnk_status lnk_paged_step_attn(const lnk_attn_desc* desc, const lnk_bf16* q_roped,
                               const int32_t* rows, const int32_t* positions,
                               const int32_t* segments, const int32_t* step_positions,
                               const int32_t* table, const lnk_bf16* k_pool,
                               const lnk_bf16* v_pool, lnk_bf16* out, const int32_t* last,
                               lnk_bf16* last_out, int32_t P, int32_t B, int32_t M,
                               void* workspace, size_t ws_bytes, int32_t* dev_status,
                               lnk_stream stream);

/*
 * lnk_paged_decode_attn_static -- lnk_paged_decode_attn without a workspace
 * argument; it allocates nothing.  (The pages have no counterpart: this is a
 * calling convention of the library, not a step of the method.)
 *
 * For callers that cannot provide scratch memory when the step runs: code run
 * by a host runtime that has reserved all device memory and forbids allocation
 * on its execution path, or a serving loop that must keep its memory footprint
 * and step latency fixed.  The decode scratch lives instead in a static device
 * array of 8 MiB inside the library, which every GPU that loads the library
 * keeps until the process exits.  Calls whose lnk_paged_workspace_size(desc, B)
 * exceeds 8 MiB return LNK_ERANGE and enqueue nothing.
 *
 * The first call on a device, made with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture.  A failed lookup returns LNK_ECUDA and is retried by the
 * next call.  Once its arguments have passed every check, a call clears the
 * array's counters on `stream` (cudaMemsetAsync) and then runs the same kernel
 * as lnk_paged_decode_attn; a call that returns an error enqueues nothing.
 * All calls share the one array: calls that may run at the same time on the
 * GPU (different streams or host threads) race and must be ordered by the
 * caller.  Arguments, layouts and errors are otherwise those of
 * lnk_paged_decode_attn (a descriptor that lnk_paged_workspace_size rejects
 * gives LNK_EINVAL).
 */
lnk_status lnk_paged_decode_attn_static(const lnk_attn_desc* desc, const lnk_bf16* q_roped,
                                        const int32_t* positions, const int32_t* table,
                                        const lnk_bf16* k_pool, const lnk_bf16* v_pool,
                                        lnk_bf16* out, int32_t B, int32_t* dev_status,
                                        lnk_stream stream);

/* ---------------------------------------------------------------------------
 * Host page allocator (lnk_pager) and page copies
 *
 * Source: "Mistral 7B Instruct v0.3", Entries table (prefill_paged): a token
 * attends over its row's pages up to its position -- "chunks, shared
 * prefixes", so rows may map the same physical pages for a common prefix.
 * The pages do not say how pages are handed out; this allocator is the
 * plainest one that supports that sharing:
 *   - free pages are handed out lowest page number first;
 *   - each page has a reference count = the number of table entries mapping it;
 *   - fork maps a new row onto the pages of another row's prefix;
 *   - before a token is written, prepare_append maps a fresh page for an
 *     unmapped logical page, and moves a row that writes into a page mapped
 *     more than once onto a fresh private page (copy on write): the caller
 *     copies the old page into the new one with lnk_paged_copy_pages before
 *     the append;
 *   - release drops a row's pages; a page whose count reaches 0 is free.
 * The pager holds host memory only (its table is exported into a caller
 * buffer for upload to the device) and is not thread-safe: serialise the
 * calls made on one pager.  Host pointers below are host memory.
 * ------------------------------------------------------------------------- */
typedef struct lnk_pager lnk_pager;

/* A pager over num_pages pages for a table of num_rows x pages_per_row, all
 * unmapped (-1).  *out receives the handle (NULL on error).  LNK_EINVAL for a
 * non-positive size, LNK_ENOSPACE if host memory runs out. */
lnk_status lnk_pager_create(int32_t num_pages, int32_t num_rows, int32_t pages_per_row, lnk_pager** out);

/* Frees the pager (NULL is ignored). */
void lnk_pager_destroy(lnk_pager* pager);

/* Maps a fresh page to every unmapped logical page of `row` covering positions
 * [0, length).  Mapped pages are left as they are (shared ones included).
 * LNK_ERANGE if length > pages_per_row * 64; LNK_ENOSPACE (nothing changed) if
 * the free pages do not suffice. */
lnk_status lnk_pager_reserve(lnk_pager* pager, int32_t row, int32_t length);

/* Maps the first ceil(length / 64) logical pages of the empty row dst_row onto
 * src_row's pages (their counts + 1); src_row must have them mapped.  A shared
 * partial last page is copied on the first write into it (prepare_append).
 * LNK_EINVAL if dst_row is not empty, src_row lacks a page, or the rows are
 * equal or out of range. */
lnk_status lnk_pager_fork(lnk_pager* pager, int32_t src_row, int32_t dst_row, int32_t length);

/* Prepares the n tokens (rows[t], positions[t]; host arrays) that the next
 * lnk_paged_append_rope will write, in order: the first token of the batch
 * that writes into a logical page maps a fresh page if it is unmapped, or
 * moves the row onto a fresh page if the page is mapped by other rows too;
 * each such move appends (old page, new page) to copy_src/copy_dst (host
 * arrays of capacity n) and *num_copies counts them.  Negative positions are
 * skipped.  LNK_EINVAL for a bad row, LNK_ERANGE for a position past the
 * table row, LNK_ENOSPACE if the free pages do not suffice; on any error
 * nothing changes. */
lnk_status lnk_pager_prepare_append(lnk_pager* pager, const int32_t* rows, const int32_t* positions, int32_t n,
                                    int32_t* copy_src, int32_t* copy_dst, int32_t* num_copies);

/* Unmaps every page of `row`; pages whose count reaches 0 become free. */
lnk_status lnk_pager_release(lnk_pager* pager, int32_t row);

/* Writes the table, [num_rows][pages_per_row] int32 (-1 = unmapped), into the
 * host buffer `table`. */
lnk_status lnk_pager_table(const lnk_pager* pager, int32_t* table);

/* Number of free pages (-1 for a NULL pager). */
int32_t lnk_pager_free_pages(const lnk_pager* pager);

/* Reference count of `page` (-1 for a NULL pager or a page out of range). */
int32_t lnk_pager_refcount(const lnk_pager* pager, int32_t page);

/* Copies pages src_pages[i] -> dst_pages[i] (device int32 arrays of n) in the
 * K and V pools (of the desc's element type), every kv head (the copy on
 * write of prepare_append).  A pair
 * with a page outside [0, num_pages) is skipped and sets LNK_DEV_BAD_PAGE in
 * *dev_status.  Pairs must not overlap (no page both a source and a target).
 * Enqueued on `stream`; call it before the append that writes the pages. */
lnk_status lnk_paged_copy_pages(const lnk_attn_desc* desc, lnk_bf16* k_pool, lnk_bf16* v_pool,
                                const int32_t* src_pages, const int32_t* dst_pages, int32_t n,
                                int32_t* dev_status, lnk_stream stream);

/* ---------------------------------------------------------------------------
 * Self-test of the bounded waits.  Every wait inside the kernels above is
 * bounded: after about two seconds it gives up, the CTA's other roles stop,
 * the kernel ORs LNK_DEV_TIMEOUT into *dev_status and returns (no trap, no
 * fault).  This call runs that path on purpose: one CTA of two warps waits on
 * pipeline barriers that nothing arrives at; the first gives up after
 * limit_ns (1 .. 2e9), the second must then stop through the CTA's abort flag
 * rather than its own two-second limit.  dev_status (device) receives
 * LNK_DEV_TIMEOUT.  LNK_EINVAL for a null status or a limit out of range.
 * ------------------------------------------------------------------------- */
lnk_status lnk_selftest_wait_timeout(int32_t* dev_status, uint64_t limit_ns, lnk_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* LNK_H */
