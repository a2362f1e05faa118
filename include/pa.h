/*
 * pa.h - C ABI of the GB300 (sm_103a) windowed prefill attention over a paged
 * int8 KV pool.
 *
 * The operation ("int8 tensor-core prefill attention", sections "Summary" and
 * "Why the attention, and why tensor cores"; window-off case in "Relation to
 * open PRs"; pool layout and StreamingLLM window in "fp16 shared-memory tiles
 * for windowed prefill attention", "Summary"):
 *
 *   for every sequence, query token t (absolute position) and q head h, with
 *   kv head g = h / (n_q_heads / n_kv_heads):
 *     key j is visible iff j <= t and, when n_win_blk > 0,
 *       j/16 < n_sink_blk  or  j/16 >= max(0, t/16 + 1 - n_win_blk)
 *     K_j = k_pool code * k_scale,  V_j = v_pool code * v_scale   (per token, per kv head)
 *     out[t][h] = softmax_j(sm_scale * <q[t][h], K_j>) . V_j     over visible j
 *
 * computed along the pages' method: per-row Q / per-token K / softmax scales
 * applied to the scores of integer-valued K codes, an online softmax over key
 * tiles that skips masked blocks, and the per-token V scale folded into P.  By
 * default the query enters the tensor core as given (bf16) and P' = p * v_scale
 * is held in fp16; the pages' per-row int8 query and u8 P grids are options
 * (PA_Q_INT8, PA_P_U8 below).
 *
 * Layouts (all row-major, C order):
 *   q, out        bf16  [total_q][n_q_heads][256]          16-byte aligned
 *   k_pool,v_pool int8  [n_pool_pages][16][n_kv_heads][256] 16-byte aligned
 *   k_scale,
 *   v_scale       fp32  [n_pool_pages][16][n_kv_heads]      4-byte aligned
 *   block_table   int32 [n_seq][max_pages_per_seq]: logical page -> pool page
 *
 * Ownership: every tensor argument is caller-owned memory; device entry points
 * take device pointers, pa_prefill_host takes host pointers.  The handle owns
 * only its workspace (widened K/V copies of the visible pages, work list,
 * error word), grown on demand and freed by pa_destroy.
 *
 * Asynchrony: pa_prefill / pa_prefill_batch only enqueue work on `stream`
 * (a cudaStream_t; NULL = legacy default stream) and return; device-side
 * failures (a bounded wait that ran out, a block-table entry outside the pool)
 * are reported by the next pa_last_error.  A handle serialises its own calls:
 * use one handle per concurrently running stream.
 *
 * Return codes: PA_OK (0) or a negative PA_E* code; pa_strerror names it.
 */
#ifndef PA_H
#define PA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_OK 0
#define PA_EINVAL (-1)    /* bad argument: shape, null pointer, alignment, range */
#define PA_EARCH (-2)     /* current device is not an sm_103 GPU */
#define PA_ECUDA (-3)     /* a CUDA runtime call or kernel launch failed */
#define PA_ETIMEOUT (-4)  /* a device-side wait ran out (see pa_options.wait_timeout_ms) */
#define PA_EBADPAGE (-5)  /* a block-table entry read was outside [0, n_pool_pages) */
#define PA_ENOMEM (-6)    /* workspace allocation failed */
#define PA_ENOSCRATCH (-7) /* pa_prefill_noalloc: the call needs more than PA_NOALLOC_SCRATCH_BYTES */

/* Query container (step "Q per-row quantise", fused into the kernel prologue). */
#define PA_Q_BF16 0  /* default: Q's bf16 values enter the MMA unchanged (no rounding; s_q = 1) */
#define PA_Q_INT8 1  /* the pages' grid: scale absmax/127, codes rint(q*127/absmax) in [-127,127] */
/* P container (step "V scale folded into P, P quantised per row"). */
#define PA_P_F16 0   /* default: P' = p * v_scale rounded to fp16 (11-bit significand) */
#define PA_P_U8 1    /* the pages' grid per row and 128-key tile: scale max/255, codes in [0,255] */

typedef struct pa_ctx* pa_handle;

typedef struct {
  int q_mode;           /* PA_Q_BF16 | PA_Q_INT8 */
  int p_mode;           /* PA_P_F16 | PA_P_U8 */
  int wait_timeout_ms;  /* bound on every device-side wait (default 2000) */
  int record_timing;    /* nonzero: time each launch with CUDA events (pa_timing) */
  int debug_stall;      /* test hook: nonzero makes the attention kernel's first wait target a
                           barrier nothing arrives at, so the bounded wait runs out, the kernel
                           exits cleanly and pa_last_error reports PA_ETIMEOUT; 0 in normal use */
  int debug_fail_host;  /* test hook: nonzero makes pa_prefill_host fail as if a CUDA call had
                           failed while it was still enqueuing (after the pool's and the first
                           chunks' copies were issued), to test that it drains its copies before
                           returning PA_ECUDA; 0 in normal use */
} pa_options;

typedef struct {
  int q_off;    /* first row of this sequence in q and out */
  int q_start;  /* absolute position of that row (tokens already cached) */
  int n_q;      /* query tokens of this sequence (>= 1) */
  int n_ctx;    /* context tokens in the pool; q_start + n_q <= n_ctx */
} pa_seq;

/* Fill *opt with the defaults (bf16 query as given, fp16 P', 2000 ms waits, no timing, no test hooks). */
void pa_default_options(pa_options* opt);

/* Create a handle bound to the current CUDA device.  head_dim must be 256 and
 * page_size 16; n_q_heads % n_kv_heads == 0 and 128 % (n_q_heads/n_kv_heads)
 * == 0; n_kv_heads <= 8.  opt may be NULL (defaults).  PA_EARCH unless the
 * device is sm_103. */
int pa_create(pa_handle* h, int n_q_heads, int n_kv_heads, int head_dim, int page_size, int n_pool_pages,
              int max_pages_per_seq, const pa_options* opt);

/* Release the handle and its workspace (synchronises the device). */
void pa_destroy(pa_handle h);

/* One sequence: queries are tokens [q_start, q_start + n_q) of a context of
 * n_ctx tokens whose pages block_table[0 .. ceil(n_ctx/16)) lists.  q and out
 * hold n_q rows.  n_win_blk <= 0 turns the window off (plain causal). */
int pa_prefill(pa_handle h, const void* q, const int8_t* k_pool, const int8_t* v_pool, const float* k_scale,
               const float* v_scale, const int32_t* block_table, int q_start, int n_q, int n_ctx, int n_sink_blk,
               int n_win_blk, float sm_scale, void* out, void* stream);

/* Several sequences in one launch.  seqs is a HOST array of n_seq entries;
 * block_table row s belongs to seqs[s]; all sequences share the pool. */
int pa_prefill_batch(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const int8_t* k_pool,
                     const int8_t* v_pool, const float* k_scale, const float* v_scale, const int32_t* block_table,
                     int n_sink_blk, int n_win_blk, float sm_scale, void* out, void* stream);

/* pa_prefill_batch with the output gate fused into the epilogue ("int8
 * tensor-core prefill attention", section "Correctness": the attention output
 * is multiplied by sigmoid(q_gate) before the next layer):
 *   out[t][h][d] = bf16( bf16(attention[t][h][d]) * sigmoid(q_gate[t][h][d]) )
 * i.e. the value a separate elementwise gate kernel would produce from the
 * ungated bf16 output.  q_gate is a device pointer, bf16 [total_q][n_q_heads]
 * [256] like q and out, 16-byte aligned, caller-owned, read once.  Errors as
 * pa_prefill_batch; PA_EINVAL for a NULL or misaligned q_gate. */
int pa_prefill_batch_gated(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const void* q_gate,
                           const int8_t* k_pool, const int8_t* v_pool, const float* k_scale, const float* v_scale,
                           const int32_t* block_table, int n_sink_blk, int n_win_blk, float sm_scale, void* out,
                           void* stream);

/* pa_prefill_batch on HOST buffers: copies the inputs to handle-owned device
 * memory, runs, copies out back and synchronises `stream`; the return value
 * includes device-side errors.  The copies overlap the computation: the pool
 * goes in first and is widened once, the query rows are split into chunks
 * (whole work units of 256 / G tokens), and while one chunk is computed on
 * `stream` the next one's q rows are copied in and the previous one's output
 * rows copied out on two copy streams the handle owns.  The result is the one
 * pa_prefill_batch gives on device copies of the same buffers.
 * Output rows that belong to no sequence are left as they were.  Pinned host
 * memory is fastest (pageable memory makes the copies synchronous).
 * Every call copies the whole pool, scales and block table in again (the
 * handle keeps no copy of host data between calls).
 * Waits: the attention launch of a chunk after the first waits on the device
 * for a flag the copy stream writes once that chunk's rows are in; that wait
 * has the same bound as every device wait (pa_options.wait_timeout_ms, 2 s by
 * default), measured from the launch's start, so a copy link slower than
 * about (chunk rows x n_q_heads x 512 bytes) per bound can end the call with
 * PA_ETIMEOUT: raise wait_timeout_ms for slow links or pageable memory.
 * Failure: once the first copy is issued, a failing CUDA call makes the
 * function wait for both copy streams and `stream` before returning its
 * error, so no copy reads the caller's buffers or writes `out` afterwards. */
int pa_prefill_host(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const int8_t* k_pool,
                    const int8_t* v_pool, const float* k_scale, const float* v_scale, const int32_t* block_table,
                    int n_sink_blk, int n_win_blk, float sm_scale, void* out, void* stream);

/* Debug (tests): 1 if the handle's two copy streams (those of
 * pa_prefill_host) have no work pending, 0 if either still has, PA_EINVAL
 * for a NULL handle, PA_ECUDA if a stream reports an error.  Does not wait. */
int pa_debug_copy_streams_idle(pa_handle h);

/* Synchronise `stream`, then report and clear the first device-side error
 * recorded since the last call (PA_ETIMEOUT, PA_EBADPAGE) or PA_ECUDA. */
int pa_last_error(pa_handle h, void* stream);

/* Launch times recorded since the last reset (needs record_timing): sums of
 * the widening pass and the attention kernel in milliseconds, and the number
 * of calls.  A pa_prefill_host call counts once; its attention time runs from
 * the end of its widening pass to the end of its last chunk, waits for the
 * chunks' rows included.  Waits for the recorded events. */
int pa_timing(pa_handle h, int reset, double* widen_ms, double* attention_ms, int* n_calls);

const char* pa_strerror(int code);

/* KV append, the step before the path ("fp16 shared-memory tiles for windowed
 * prefill attention", "Summary": K and V live in an int8 paged pool with
 * per-token, per-kv-head fp32 scales): the K and V rows of n_new new tokens,
 * positions [tok_start, tok_start + n_new) of one sequence, are quantised and
 * written into the pool.  Each (token, kv head) row of 256 values gets its own
 * symmetric scale absmax/127 and codes rint(x/scale), half to even, clamped to
 * [-127, 127]; all decisions in fp32 with correctly rounded divisions; an
 * all-zero row gets scale 0 and codes 0.  Row (token t, head g) goes to page
 * block_table_row[t / 16], slot t % 16, i.e. k_pool[page][t % 16][g][:] and
 * k_scale[page][t % 16][g] (likewise V).
 *   k_new, v_new     device bf16 [n_new][n_kv_heads][256], 16-byte aligned
 *   block_table_row  device int32, the sequence's pages (>= ceil((tok_start +
 *                    n_new) / 16) entries, at most max_pages_per_seq)
 *   pools, scales    device, the layouts of pa_prefill; written in place
 * Asynchronous on `stream`; no other slot is touched.  A page entry outside
 * [0, n_pool_pages) is never dereferenced: its rows are skipped and
 * pa_last_error reports PA_EBADPAGE.  PA_EINVAL for bad pointers, alignment or
 * a range past max_pages_per_seq pages.  Inputs must be finite. */
int pa_kv_append(pa_handle h, const void* k_new, const void* v_new, int n_new, int tok_start,
                 const int32_t* block_table_row, int8_t* k_pool, int8_t* v_pool, float* k_scale, float* v_scale,
                 void* stream);

/* Decode: one new query token per sequence against the same pool and mask
 * (the decode path that shares the prefill's window selection, "int8
 * tensor-core prefill attention", sections "Why the attention, and why tensor
 * cores" and "Relation to open PRs").  seqs[s] must have n_q == 1 and q_start
 * == n_ctx - 1: the token is the context's last; its row in q and out is
 * seqs[s].q_off; block_table row s holds its pages.  Layouts as pa_prefill_batch
 * (q, out bf16 [rows][n_q_heads][256]).  The visible 16-token blocks of all
 * (sequence, kv head) pairs are split into runs of equal cost (pa_decode_plan)
 * computed in parallel and merged on the device; q, the pool and P' stay in exact or fp16
 * containers (the bf16 query scaled per row by a power of two, codes as exact
 * fp16, P' = p * v_scale in fp16, fp32 accumulation).  One launch per 512
 * sequences, the sequence table carried in its parameters (no host-to-device
 * copy, no host wait).  Needs n_q_heads / n_kv_heads <= 8 and fewer than
 * 2^30 visible blocks x kv heads per 512 sequences (PA_EINVAL otherwise).  Calls on one handle share its work
 * buffers: issue them on one stream (calls that overlap on the GPU race).
 * Asynchronous; device errors (PA_EBADPAGE for a page entry outside the pool,
 * whose block is skipped) through pa_last_error. */
int pa_decode(pa_handle h, int n_seq, const pa_seq* seqs, const void* q, const int8_t* k_pool, const int8_t* v_pool,
              const float* k_scale, const float* v_scale, const int32_t* block_table, int n_sink_blk, int n_win_blk,
              float sm_scale, void* out, void* stream);

/* Host-only, no GPU needed: how pa_decode splits the work of one launch (the
 * first min(n_seq, 512) sequences) when `slots` of its CTAs run at once (SMs x
 * CTAs per SM; two per SM on a GB300).  The launch's (sequence, kv head)
 * pairs, sequence-major, laid end to end give a list of *total_blocks visible
 * 16-token blocks; CTA c computes the run from its first block to the next
 * CTA's.  *listed = 1: one wave of runs of equal cost (blocks + 16 for every
 * pair after a run's first), at most *per_cta (the budget, <= 128); 0: runs of
 * *per_cta blocks over whole waves.  runs_out (may be NULL) receives *n_cta
 * entries of int32[3] = {first block, its sequence, the CTA's partial slot in
 * that block's pair (the CTAs before it in the pair)}; *max_slots = the most
 * CTAs one pair's blocks meet.  PA_EINVAL for bad shapes, a sequence that is
 * not a decode query (n_q == 1, q_start == n_ctx - 1), or cap < *n_cta. */
int pa_decode_plan(int n_kv_heads, int slots, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
                   int32_t* runs_out, int cap, int* n_cta, int* per_cta, int* max_slots, int* listed,
                   long long* total_blocks);

/* Query rows per work unit: the G = n_q_heads / n_kv_heads q heads of one kv
 * head times PA_UNIT_ROWS / G consecutive tokens starting on a multiple of
 * PA_UNIT_ROWS / G.  One unit is one 256-row tensor-core tile computed by a
 * pair of SMs (128 rows each), so every row of a unit shares the keys its
 * tiles visit: the union of the visible key blocks of the unit's query blocks. */
#define PA_UNIT_ROWS 256

/* Host-only planning, no GPU needed: the work units of a call, longest first
 * (the launch then hands them to the kernel's SM pairs: pa_plan_pairs).
 * units_out (may be NULL) receives up to cap entries of int32[4] = {sequence,
 * kv head, first token, key tiles}.  Outputs: unit count, total key tiles,
 * widened rows. */
int pa_plan(int n_q_heads, int n_kv_heads, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
            int32_t* units_out, int cap, int* n_units, long long* n_tiles, int* n_widened_rows);

/* Host-only, no GPU needed: pa_plan's units as a launch hands them to n_pairs
 * SM pairs (the attention kernel runs min(units, 76) pairs on a 152-SM
 * GB300): longest first, each to the pair whose work so far (key tiles, plus
 * two for each unit change) is least, ties to the lowest pair; then laid out
 * pair by pair.  units_out (int32 [n_units][4], as pa_plan; may be NULL when
 * cap is 0) receives them in that layout, pair_off (int32 [n_pairs + 1]) each
 * pair's first unit and, last, the count.  PA_EINVAL for bad shapes,
 * n_pairs < 1, or cap < the unit count when units_out is given. */
int pa_plan_pairs(int n_q_heads, int n_kv_heads, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
                  int n_pairs, int32_t* units_out, int cap, int32_t* pair_off, int* n_units);

/* Host-only, no GPU needed: the chunks pa_prefill_host cuts the query rows of
 * a call into, when the attention kernel runs n_pairs CTA pairs at once (76 on
 * a 152-SM GB300).  The rows of the sequences laid end to end (seqs order) go
 * in chunks of work units counted in waves (a wave: one unit per pair): one
 * wave first, one wave last (or less: the remainder), two waves in between;
 * a boundary inside a sequence falls on a multiple of
 * PA_UNIT_ROWS / G tokens (absolute position), so every work unit lies in one
 * chunk.  chunk_end (may be NULL) receives up to cap increasing row counts,
 * the last = the total rows; *n_chunks the count.  PA_EINVAL for bad shapes
 * or cap < the count. */
int pa_host_chunks(int n_q_heads, int n_kv_heads, int n_seq, const pa_seq* seqs, int n_pairs, long long* chunk_end,
                   int cap, int* n_chunks);

/* Debug (tests): run the widening pass, then export sequence `seq`'s widened
 * rows: k_out/v_out int8 [n_kv_heads][n_rows][256], ks_out/vs_out fp32
 * [n_kv_heads][n_rows], tok_out int32 [n_rows] (logical token of each row, -1
 * past n_ctx); all device pointers with room for `cap` rows.  *n_rows (host)
 * receives the row count.  Synchronous. */
int pa_debug_gather(pa_handle h, int n_seq, const pa_seq* seqs, const int8_t* k_pool, const int8_t* v_pool,
                    const float* k_scale, const float* v_scale, const int32_t* block_table, int n_sink_blk,
                    int n_win_blk, int seq, int8_t* k_out, int8_t* v_out, float* ks_out, float* vs_out,
                    int32_t* tok_out, int cap, int* n_rows, void* stream);

/* Debug (tests): for every work unit, the key blocks its tiles visit
 * (unit_blocks int32 [n_units][cap], -1 padded) and per row the number of keys
 * the kernel's mask admits (row_counts int32 [n_units][PA_UNIT_ROWS]); device
 * pointers.
 * units_out (host int32 [n_units][4], as pa_plan) names each unit.  Synchronous. */
int pa_debug_maskset(pa_handle h, int n_seq, const pa_seq* seqs, int n_sink_blk, int n_win_blk,
                     int32_t* row_counts, int32_t* unit_blocks, int cap, int32_t* units_out, int units_cap,
                     int* n_units, void* stream);

/* Debug (tests): the per-row int8 query grid of the fused prologue ("int8
 * tensor-core prefill attention", section "Why the attention, and why tensor
 * cores": Q is quantised per query row with one scale per row), run by the
 * attention kernel's own quantiser on n_rows rows staged as its Q tile holds
 * them.  Per row: absmax over the 256 values, scale = absmax / 127 and codes
 * rint(q * (127 / absmax)) half to even, clamped to [-127, 127], every
 * decision in fp32 (IEEE divisions); an all-zero row gets scale 0 and codes 0.
 *   q_rows  device bf16 [n_rows][256], 16-byte aligned (caller-owned, read)
 *   codes   device int8 [n_rows][256], 4-byte aligned (written)
 *   scales  device fp32 [n_rows] (written)
 * Synchronous on `stream`.  PA_EINVAL for a negative count, NULL or misaligned
 * pointers; PA_ECUDA if the launch fails. */
int pa_debug_qcodes(const void* q_rows, int n_rows, int8_t* codes, float* scales, void* stream);

/* Allocation-free variant of pa_prefill (one sequence, default
 * containers).  The pages have no counterpart of this entry point: it exists
 * for callers that may not call cudaMalloc / cudaFree, for example an engine
 * that has reserved nearly all device memory for its own KV-cache pool and
 * accounts for every byte, or code on a latency-critical path where an
 * allocation, which can synchronise the device, is not allowed.
 *
 * It takes no handle and allocates nothing: its scratch (widened K/V copies
 * of the visible pages, scales, work list, error word) lives in one static
 * device array of PA_NOALLOC_SCRATCH_BYTES that every GPU loading this
 * library holds until the process exits.  Arguments and layouts are those of
 * pa_create + pa_prefill.  A call whose visible context does not fit
 * (widened rows x n_kv_heads x 1032 bytes plus a 1 MiB work list) returns
 * PA_ENOSCRATCH before touching the GPU; with the 32 MiB array that is about
 * 32000 token-heads, e.g. 16000 visible tokens for 2 kv heads.
 *
 * All calls share the one array and each call clears what must start at
 * zero, so calls on different streams, or from different threads, that
 * overlap on the GPU race and corrupt each other: serialise them.
 *
 * Set-up: the first call on a device (and the first after that device's
 * context was reset, which reloads the module) looks up the array's device
 * address with cudaGetSymbolAddress and reads the device's compute capability
 * and SM count, with that device current; that first call should come before
 * any stream capture.  Later calls reuse what it found.
 *
 * The work list has the order pa_plan gives (longest units first).  The call
 * is synchronous: after enqueuing its kernels on `stream` it reads this
 * call's device-side status word on `stream` and waits for `stream` alone,
 * returning PA_ETIMEOUT or PA_EBADPAGE from the device.  PA_EINVAL for the
 * argument errors of pa_create / pa_prefill, including q_start + n_q or n_ctx
 * above 2^30. */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
int pa_prefill_noalloc(int n_q_heads, int n_kv_heads, int n_pool_pages, int max_pages_per_seq, const void* q,
                       const int8_t* k_pool, const int8_t* v_pool, const float* k_scale, const float* v_scale,
                       const int32_t* block_table, int q_start, int n_q, int n_ctx, int n_sink_blk, int n_win_blk,
                       float sm_scale, void* out, void* stream);

/* Debug export (tests only; like pa_prefill_noalloc, the pages have no
 * counterpart): copies the work list the last pa_prefill_noalloc call on the
 * current device built in its scratch array into units_out (host int32
 * [n_units][4] = {sequence (0), kv head, first token, key tiles}, the layout
 * of pa_plan's units).  Synchronous on `stream`; call it after that call and
 * before any other on the device.  PA_EINVAL for n_units outside (0, the
 * array's work-list capacity] or a NULL pointer. */
int pa_debug_noalloc_units(int n_units, int32_t* units_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
