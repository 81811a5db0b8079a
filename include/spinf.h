/*
 * spinf.h -- C ABI of the branch-packed scoring hot path for GB300 (sm_103a).
 *
 * The problem, as the pages state it ("spinf-serve 0.1.1", PyPI project page,
 * sections "What it does" and "Install and run"): a request holds contents and,
 * per content, questions; a question is a template that ends where the answer
 * goes ({?}) with the options to score there.  The engine reads each content
 * once, lays every question out as a branch of the same packed pass, and
 * returns per option its log-probability, its probability renormalised over the
 * options (p), the same on empty content (the floor), and the mass that went
 * outside the options (residual).  There is no tokenizer here: every text is
 * given as token ids.
 *
 * The path, in call order:
 *   spinf_pack_plan         host: inputs -> packed passes of <= token_budget rows
 *   spinf_plan_upload       host -> device: one pass's descriptors
 *   spinf_branch_attention  device: tree-masked GQA attention over the pass
 *   spinf_score             device: lm-head at slot rows, full-vocabulary
 *                           log-sum-exp, option-token log-probabilities
 *                           (spinf_score_extract: also the top tokens of
 *                           searched slots, in the same read of the lm head)
 *   spinf_collect           host: per option lp, p, residual and floor
 *                           (spinf_collect_extract: searched-slot answers)
 *
 * Conventions for every call:
 *   - Status codes only; nothing throws across this boundary.  The text of the
 *     last error of the calling thread is returned by spinf_last_error().
 *   - The caller owns every device buffer (passed as raw device pointers) and
 *     every host array it passes in.  The planner copies what it keeps.  A plan
 *     owns its host tables and the device copies made by spinf_plan_upload
 *     until spinf_plan_free.
 *   - Device calls are asynchronous on the given stream (NULL = legacy default
 *     stream) and allocate nothing: scratch memory is the caller's workspace.
 *   - Device buffers must be 16-byte aligned; all device tensors are dense,
 *     row-major, tokens the slowest dimension.
 *   - There is no CPU fallback: a device call on a machine without an sm_103a
 *     GPU returns SPINF_E_CUDA.
 *   - A plan may be used from several host threads: the per-pass caches built
 *     on first use (window schedules, rotary tables) are guarded by a lock in
 *     the plan; uploads (spinf_plan_upload*) and spinf_plan_free are not, and
 *     must not overlap other calls on the same plan.
 */
#ifndef SPINF_H
#define SPINF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                      /* the same type as cudaStream_t */
typedef struct CUstream_st* spinf_stream;

typedef enum {
    SPINF_OK = 0,
    SPINF_E_INVALID = 1,        /* malformed request or argument */
    SPINF_E_LIMIT = 2,          /* a limit of spinf_plan_opts exceeded */
    SPINF_E_NOMEM = 3,          /* host or device allocation failed, or workspace too small */
    SPINF_E_CUDA = 4,           /* a CUDA runtime call failed (no device, launch error, ...) */
    SPINF_E_UNSUPPORTED = 5,    /* a shape or dtype this library does not implement */
    SPINF_E_DEVICE_TIMEOUT = 6, /* a bounded device wait ran out (reported by spinf_device_status) */
    SPINF_E_DEVICE_CHECK = 7    /* a device-side descriptor check failed */
} spinf_status;

enum { SPINF_DTYPE_BF16 = 0, SPINF_DTYPE_E4M3 = 1 };

/* Question kinds ("spinf-serve 0.1.1" PyPI page, "What it does"; man page,
 * DESCRIPTION): a scored template ends in {?} and carries options; a searched
 * slot ({*} text, {n} numbers, {$} amounts) carries none and returns the most
 * likely next tokens with their probabilities. */
enum { SPINF_Q_SCORED = 0, SPINF_Q_SEARCHED = 1 };

/* A token-id array (host memory). */
typedef struct {
    const int32_t* ids;
    int32_t n;
} spinf_tokens;

/* One question: template tokens up to and including the last token before the
 * slot.  kind SPINF_Q_SCORED (0, so a zeroed struct is a scored question): the
 * options to score at the slot (1 to max_option_tokens tokens each; no
 * duplicates).  kind SPINF_Q_SEARCHED: no options (n_options 0); the slot
 * returns its extract_k most likely tokens among the allowed-token set number
 * token_set given at scoring time (-1: every token).  Decoding a longer answer
 * appends the chosen tokens to the template and plans again. */
typedef struct {
    spinf_tokens tmpl;
    const spinf_tokens* options;
    int32_t n_options;
    int32_t kind;
    int32_t token_set;
} spinf_question;

/* A question grid ("spinf-serve 0.1.1" PyPI page, "What it does": placeholders
 * turn one template into a grid of questions).  The template is
 *   segments[0] v_0 segments[1] v_1 ... v_{n-1} segments[n],  n = n_placeholders,
 * v_i one of placeholder i's values; the grid stands for one question per
 * combination of values, the first placeholder varying slowest, each with the
 * grid's options (kind SPINF_Q_SCORED) or a searched slot (SPINF_Q_SEARCHED,
 * token_set).  Segments and values may be empty token arrays; every placeholder
 * needs at least one value. */
typedef struct {
    const spinf_tokens* segments;   /* [n_placeholders + 1] */
    int32_t n_placeholders;         /* >= 0 */
    const spinf_tokens* values;     /* every placeholder's values, placeholder by placeholder */
    const int32_t* n_values;        /* [n_placeholders], each >= 1 */
    const spinf_tokens* options;
    int32_t n_options;
    int32_t kind;
    int32_t token_set;
} spinf_grid;

/* One input: a content (may be empty) read once, its questions, then the cells
 * of its grids (grid by grid; a zeroed grids field means none).  Grid cells are
 * questions like any other: they are numbered after the input's own questions
 * and count toward max_prompts_per_input. */
typedef struct {
    spinf_tokens content;
    const spinf_question* questions;
    int32_t n_questions;
    const spinf_grid* grids;
    int32_t n_grids;
} spinf_input;

/* Planner options.  Defaults (spinf_plan_opts_default) follow the man page
 * ("spinf-serve", linuxcommandlibrary, PARAMETERS): --token-budget 16384,
 * --max-content-tokens 4096, --max-query-tokens 256, --max-options 1000,
 * --max-option-tokens 5, --max-prompts-per-input 10000.  --max-tokens has no
 * printed default; it defaults to 2,000,000 (the per-request processed-token
 * limit on the same page). */
typedef struct {
    int32_t token_budget;           /* rows per packed pass */
    int32_t max_tokens;             /* largest single input: content plus its laid-out questions */
    int32_t max_content_tokens;
    int32_t max_query_tokens;       /* template length */
    int32_t max_options;
    int32_t max_option_tokens;
    int32_t max_prompts_per_input;  /* questions per input */
    int32_t floors;                 /* 1: add one floor input per distinct (template, options) */
    spinf_tokens floor_prefix;      /* content of every floor input (default: empty) */
    int32_t vocab;                  /* > 0: reject token ids outside [0, vocab) */
    int32_t extract_k;              /* tokens returned per searched slot, 1..16 (default 8) */
} spinf_plan_opts;

typedef struct spinf_plan spinf_plan;

/* Read-only host views of one packed pass (valid until spinf_plan_free). */
typedef struct {
    int32_t T;          /* rows holding tokens */
    int32_t T_pad;      /* T rounded up to a multiple of 128; device tensors have T_pad rows */
    int32_t n_qtiles;   /* T_pad / 128 */
    int32_t n_sched;    /* entries of tile_kv */
    int32_t M;          /* scoring rows (slots and option-prefix rows) */
    int32_t G;          /* gathered option tokens */
    int32_t n_units;    /* laid-out inputs (chunks of user inputs, then floors) */
    const int32_t* tok;       /* [T_pad] token id per row (0 on pad rows) */
    const int32_t* parent;    /* [T_pad] previous row on the root path, -1 at a root or pad */
    const int32_t* pos;       /* [T_pad] depth on the root path (position id) */
    const int32_t* end;       /* [T_pad] key k is visible to rows k <= q < end[k] */
    const int32_t* anchor;    /* [T_pad] first row of the row's input (pad: itself) */
    const int32_t* tile_ptr;  /* [n_qtiles + 1] CSR of the KV-tile schedule */
    const int32_t* tile_kv;   /* [n_sched] first row of each scheduled 128-row KV tile */
    const int32_t* tile_len;  /* [n_sched] keys of that tile that belong to its input (1..128) */
    const int32_t* slot_row;  /* [M] packed row of each scoring row, ascending */
    const int32_t* gather_m;  /* [G] scoring-row index of each option token */
    const int32_t* gather_tok;/* [G] option token id; order: unit, question, option, token */
    const int32_t* unit_start;/* [n_units + 1] first row of each unit, then T */
    const int32_t* unit_source;/* [n_units] user input index, or -1 for a floor */
    const int32_t* row_runs;  /* [T_pad][8] each row's visible keys (its root path) as up to four
                                 runs [lo, hi) of consecutive rows, nearest first, unused runs
                                 (0, 0); lo of the first run is -1 when the path has more runs */
    int32_t X;                /* searched slots of the pass */
    const int32_t* x_m;       /* [X] scoring-row index of each searched slot, in layout order */
    const int32_t* x_set;     /* [X] its allowed-token set (-1: every token) */
} spinf_pass_info;

/* Per-option and per-question results, caller-owned host arrays (fp64).
 * Options are numbered input by input, question by question, in the order
 * given; questions likewise.  Floor fields are NaN when floors are off. */
typedef struct {
    double* option_lp;        /* [n_options] sum of the option's token log-probabilities */
    double* option_p;         /* [n_options] exp(lp) renormalised over the question's options */
    double* option_floor_lp;  /* [n_options] the same question on empty content */
    double* option_floor_p;   /* [n_options] */
    double* residual;         /* [n_questions] 1 - sum of exp(lp) over the options */
    double* floor_residual;   /* [n_questions] */
} spinf_result;

/* Fill *opts with the defaults above. */
void spinf_plan_opts_default(spinf_plan_opts* opts);

/* Lay inputs out in packed passes ("spinf-serve 0.1.1" PyPI page, "What it does"
 * and "Speed and scale": the content once, every question a branch that sees its
 * own content and itself, never a sibling or another input; passes of 16k rows).
 *
 * Layout of one input: content rows, then per question its template rows, then
 * the rows of its option trie (proper prefixes of options, pre-order, children
 * in order of first insertion).  Floors (one per distinct question) follow all
 * user inputs.  Inputs larger than token_budget are split into chunks (the full
 * content plus a greedy run of questions); packing is next-fit.  The KV-tile
 * schedule of each 128-row Q tile lists, per intersecting input in layout order,
 * the 128-row KV tiles anchored at that input's first row that hold a key
 * visible to some row of the tile; a tile's keys beyond its input's last row
 * (tile_len) are not part of it, they are seen through their own input's tiles.
 *
 * A searched slot lays out its template rows only; its last template row is a
 * scoring row; it gets no floor.
 *
 * inputs: host array of n_inputs (n_inputs >= 0); opts: NULL for defaults.
 * On success *out owns a new plan.  Errors: SPINF_E_INVALID (empty template,
 * empty or duplicate option, token id out of range, empty input, a scored
 * question without options, a searched slot with options or token_set < -1,
 * extract_k outside 1..16, an unknown kind, a grid placeholder without values),
 * SPINF_E_LIMIT (a limit exceeded -- grid cells included --, or a content and one
 * question do not fit a pass), SPINF_E_NOMEM. */
spinf_status spinf_pack_plan(const spinf_input* inputs, int32_t n_inputs,
                             const spinf_plan_opts* opts, spinf_plan** out);

int32_t spinf_plan_num_passes(const spinf_plan* plan);

/* Host views of pass `pass`.  SPINF_E_INVALID for a bad index. */
spinf_status spinf_plan_pass_info(const spinf_plan* plan, int32_t pass, spinf_pass_info* out);

/* The KV-tile schedule of pass `pass` for a sliding window `window` > 0 (what
 * spinf_branch_attention runs with that window): the window-free schedule without the
 * tiles in which no row of the Q tile sees any of the tile's keys within the window
 * (pos[q] - pos[k] < window).  Skipping such a tile changes no bit of the result: it
 * is masked for every row.  Built on first use and kept by the plan; host views valid
 * until spinf_plan_free.  SPINF_E_INVALID for a bad pass, window <= 0 or NULL outputs. */
spinf_status spinf_plan_window_schedule(const spinf_plan* plan, int32_t pass, int32_t window,
                                        const int32_t** tile_ptr, const int32_t** tile_kv,
                                        const int32_t** tile_len, int32_t* n_sched);

/* The KV-tile schedule spinf_branch_attention runs for pass `pass`, window `window`
 * (0: none) and tiles of `key_tile` keys: 128, or 64 (what d_head 256 runs: each
 * input-anchored 128-key tile of the planner taken as its two 64-key halves).  A tile
 * stays iff some row of its Q tile sees one of its keys (k <= q < end[k], and
 * pos[q] - pos[k] < window when window > 0), in the planner's order; with window 0 and
 * key_tile 128 this is the planner's own schedule.  tile_ptr has n_qtiles + 1 entries
 * (spinf_pass_info); tile_kv / tile_len have *n_sched (first key, key count).  Built on
 * first use and kept by the plan; host views valid until spinf_plan_free.
 * SPINF_E_INVALID for a bad pass, window < 0, key_tile not 64 or 128, or NULL outputs. */
spinf_status spinf_plan_tile_schedule(const spinf_plan* plan, int32_t pass, int32_t window, int32_t key_tile,
                                      const int32_t** tile_ptr, const int32_t** tile_kv,
                                      const int32_t** tile_len, int32_t* n_sched);

/* spinf_plan_tile_schedule for Q tiles of `q_rows` rows: 128 (as above), or 64 (what
 * d_head 256 runs when a kv head serves two query heads: a 64-row Q tile of both heads
 * fills the MMA's 128 rows).  tile_ptr has T_pad / q_rows + 1 entries.  SPINF_E_INVALID
 * also for q_rows not 64 or 128. */
spinf_status spinf_plan_tile_schedule_q(const spinf_plan* plan, int32_t pass, int32_t window, int32_t key_tile,
                                        int32_t q_rows, const int32_t** tile_ptr, const int32_t** tile_kv,
                                        const int32_t** tile_len, int32_t* n_sched);

/* Number of user questions and options over the whole request (sizes of spinf_result). */
spinf_status spinf_plan_counts(const spinf_plan* plan, int64_t* n_questions, int64_t* n_options);

/* Number of searched slots over the whole request and the plan's extract_k
 * (spinf_collect_extract writes n_extract x extract_k answers). */
spinf_status spinf_plan_extract_counts(const spinf_plan* plan, int64_t* n_extract, int32_t* extract_k);

/* Copy pass `pass`'s descriptors to the current device (allocated once per pass
 * and kept by the plan; later calls are no-ops).  The allocation is synchronous;
 * the copy is enqueued on `stream` from a host buffer the plan keeps, so kernels
 * of this pass must run on `stream` or after it. */
spinf_status spinf_plan_upload(spinf_plan* plan, int32_t pass, spinf_stream stream);

/* Bytes of device memory that spinf_plan_upload_to needs for pass `pass` (0 for a
 * bad plan or index).  The pages have no counterpart: it serves callers that keep
 * one device buffer across requests instead of allocating per plan. */
size_t spinf_plan_descriptor_bytes(const spinf_plan* plan, int32_t pass);

/* spinf_plan_upload into caller-owned device memory: `buffer` (256-byte aligned,
 * >= spinf_plan_descriptor_bytes) receives the descriptors and, for the first pass
 * uploaded this way, the plan's device error word.  No allocation; the copy is
 * enqueued on `stream`.  The buffer must stay valid, and must not be reused by
 * another plan, until the last kernel of this plan that reads it has finished;
 * spinf_plan_free does not free it.  SPINF_E_INVALID for a NULL, misaligned or
 * short buffer, or for a pass already uploaded. */
spinf_status spinf_plan_upload_to(spinf_plan* plan, int32_t pass, void* buffer, size_t bytes,
                                  spinf_stream stream);

/* spinf_plan_upload_to, with the copy made from caller-owned page-locked host memory
 * `staging` (cudaHostAlloc / cudaHostRegister; >= spinf_plan_descriptor_bytes): the
 * descriptors are written there and the call returns as soon as the copy is enqueued.
 * From pageable memory (the plan's own staging) the call returns only once the driver
 * has staged the copy, behind every transfer already queued on the copy engine, which
 * stalls a caller that overlaps the next request's activation copies with this one's
 * kernels.  `staging` must not be written again until the copy has completed on
 * `stream`; it stays the caller's.  SPINF_E_INVALID as for spinf_plan_upload_to, and for
 * a NULL, short or pageable staging buffer.  The pages have no counterpart: it serves
 * pipelined callers. */
spinf_status spinf_plan_upload_pinned(spinf_plan* plan, int32_t pass, void* buffer, size_t bytes,
                                      void* staging, size_t staging_bytes, spinf_stream stream);

/* Tree-masked GQA attention over one packed pass ("spinf-serve 0.1.1",
 * "Speed and scale": one pass reads each content once, its questions branch off it).
 *
 * For every row q < T and query head h (kv head g = h * Hkv / Hq):
 *   o[q,h,:] = sum_k softmax_k(scale * q[q,h,:] . k[k,g,:]) v[k,g,:]
 * over the keys k visible to q: k <= q < end[k], and, when window > 0,
 * pos[q] - pos[k] < window.  Pad rows (q >= T) are written as zeros.
 *
 * q, o: device [T_pad, Hq, d_head] bf16; k, v: device [T_pad, Hkv, d_head] bf16.
 * d_head in {64, 128, 256}; Hq a multiple of Hkv; scale <= 0 means 1/sqrt(d_head).
 * Accumulation is fp32.  Key tiles are anchored at each input's first row and
 * visited in a fixed order, so a row's output is bit-identical whatever else is
 * packed in the pass.  The pass must have been uploaded.
 * Errors: SPINF_E_INVALID (pointers, alignment, not uploaded),
 * SPINF_E_UNSUPPORTED (d_head), SPINF_E_CUDA (launch). */
spinf_status spinf_branch_attention(const spinf_plan* plan, int32_t pass,
                                    const void* q, const void* k, const void* v, void* o,
                                    int32_t n_q_heads, int32_t n_kv_heads, int32_t d_head,
                                    float scale, int32_t window, spinf_stream stream);

/* Bytes of device workspace spinf_score needs for this pass and shape. */
size_t spinf_score_workspace_bytes(const spinf_plan* plan, int32_t pass,
                                   int32_t vocab, int32_t d_model, int32_t w_dtype);

/* Slot scoring ("spinf-serve 0.1.1", "What it does"; man page, --lm-head f32out).
 *
 * For every scoring row m (packed row slot_row[m]):
 *   z[m, v]    = hidden[slot_row[m], :] . w[v, :]                       (fp32 accumulate)
 *   row_lse[m] = log sum_v exp(z[m, v])        over the whole vocabulary
 *   token_lp[g]= z[gather_m[g], gather_tok[g]] - row_lse[gather_m[g]]
 * Logits never leave the chip.  With w_dtype SPINF_DTYPE_E4M3 the weights are
 * e4m3 codes with one fp32 scale per vocabulary row (w_scale[V]), the hidden
 * row is quantised to e4m3 with scale absmax/448 (fp32 division, round to
 * nearest even, saturating), and z = scale_row * w_scale[v] * (codes . codes).
 *
 * hidden: device [T_pad, d_model] bf16; w: device [vocab, d_model] bf16 or e4m3;
 * w_scale: device [vocab] fp32, 16-byte aligned (NULL for bf16); row_lse: device [M] fp32;
 * token_lp: device [G] fp32; workspace: device, >= spinf_score_workspace_bytes.
 * d_model a multiple of 16.  The vocabulary is reduced in a fixed chunk order,
 * so results do not depend on M or on the other rows of the pass.
 * Errors: SPINF_E_INVALID, SPINF_E_NOMEM (workspace too small),
 * SPINF_E_UNSUPPORTED (d_model, dtype), SPINF_E_CUDA. */
spinf_status spinf_score(const spinf_plan* plan, int32_t pass,
                         const void* hidden, const void* w, const float* w_scale, int32_t w_dtype,
                         int32_t d_model, int32_t vocab,
                         float* row_lse, float* token_lp,
                         void* workspace, size_t workspace_bytes, spinf_stream stream);

/* At most this many passes in one spinf_score_passes call. */
#define SPINF_SCORE_MAX_PASSES 32
/* What a pass's hidden buffer holds in spinf_score_passes: every packed row
 * [T_pad, d_model] (the slot rows are read at slot_row[m]), or only the scoring
 * rows [M, d_model], row m being the hidden state of the pass's scoring row m
 * (the rows spinf_plan_pass_info lists in slot_row, in that order). */
#define SPINF_HIDDEN_PASS_ROWS 0
#define SPINF_HIDDEN_SLOT_ROWS 1

/* Bytes of device workspace spinf_score_passes needs for these passes (0 for an
 * invalid list). */
size_t spinf_score_passes_workspace_bytes(const spinf_plan* plan, int32_t n_passes, const int32_t* passes,
                                          int32_t vocab, int32_t d_model, int32_t w_dtype);

/* spinf_score over several passes of one plan in one sweep of the lm head
 * ("spinf-serve 0.1.1", "What it does"; man page, --lm-head f32out).  The
 * scoring rows of the listed passes are scored as one list of rows: every
 * lm-head tile is read once for all of them, and only the last 128-row tile of
 * the list is padded (one call per pass pads every pass's last tile and reads
 * the whole head once per pass).  Each row's results are bit-identical to
 * those of spinf_score on its own pass: a row's logits, log-sum-exp and token
 * log-probabilities are computed by the same tile code in the same fixed order
 * whatever other rows share the call.
 *
 * passes: host [n_passes] distinct pass indices, each uploaded;
 * hidden, row_lse, token_lp: host arrays of n_passes device pointers, entry b
 * for pass passes[b]: hidden bf16 [T_pad, d_model] (hidden_rows
 * SPINF_HIDDEN_PASS_ROWS) or [M, d_model] (SPINF_HIDDEN_SLOT_ROWS: a caller
 * that has only the scoring rows, or copies only those to the device, passes
 * them compacted), row_lse fp32 [M], token_lp fp32 [G];
 * w, w_scale, w_dtype, d_model, vocab as for spinf_score;
 * workspace: device, >= spinf_score_passes_workspace_bytes.  Searched slots of
 * these passes get their row_lse but no answers (spinf_score_extract gives
 * those).  1 <= n_passes <= SPINF_SCORE_MAX_PASSES, else SPINF_E_INVALID /
 * SPINF_E_LIMIT; other errors as spinf_score. */
spinf_status spinf_score_passes(const spinf_plan* plan, int32_t n_passes, const int32_t* passes,
                                const void* const* hidden, int32_t hidden_rows,
                                const void* w, const float* w_scale, int32_t w_dtype,
                                int32_t d_model, int32_t vocab, float* const* row_lse, float* const* token_lp,
                                void* workspace, size_t workspace_bytes, spinf_stream stream);

/* Device buffers of the searched-slot answers of one pass. */
typedef struct {
    const uint32_t* token_sets;  /* device [n_sets][ceil(vocab / 32)]: bit (v % 32) of word v / 32 set
                                    means token v is allowed; may be NULL when n_sets is 0 */
    int32_t n_sets;              /* every x_set of the pass must be < n_sets */
    int32_t* top_tok;            /* device [X][extract_k]: tokens, most likely first (ties: lower id
                                    first); -1 past the end of a set with fewer allowed tokens */
    float* top_lp;               /* device [X][extract_k]: z - row_lse of each token (-inf past the end) */
} spinf_extract_out;

/* spinf_score plus the searched slots of the pass, read from the same pass over
 * the lm head ("spinf-serve 0.1.1", "What it does": extraction rides the same
 * read; the most likely answers with their probabilities).  For searched slot x
 * (scoring row x_m[x]) the extract_k allowed tokens with the largest z, in
 * descending z and ascending id on ties, and their z - row_lse.  Each CTA of the
 * lm-head kernel keeps the best extract_k of its 256-token tile per searched row;
 * a merge kernel orders the tiles' candidates.  The answer is a function of the
 * row's own values only.  ex NULL, or a pass without searched slots: exactly
 * spinf_score.  Workspace: spinf_score_workspace_bytes (it includes the
 * candidates).  Errors: those of spinf_score, and SPINF_E_INVALID for NULL
 * outputs, an x_set >= n_sets or NULL token_sets when a set is named. */
spinf_status spinf_score_extract(const spinf_plan* plan, int32_t pass,
                                 const void* hidden, const void* w, const float* w_scale, int32_t w_dtype,
                                 int32_t d_model, int32_t vocab,
                                 float* row_lse, float* token_lp, const spinf_extract_out* ex,
                                 void* workspace, size_t workspace_bytes, spinf_stream stream);

/* ---- Decoding steps of searched slots on the pass's cached keys and values. ---- */

/* Attention of decode rows of searched slots ("spinf-serve 0.1.1" PyPI, "What it does"
 * and "Speed and scale": extraction slots are decoded on the same read, the content and
 * the questions are not read again).  Decode row r extends the root path of pass row
 * anchor[r] (a searched slot's row) by the tokens of its chain: parent[r] is an earlier
 * decode row of the same chain (same anchor), or < 0 for the chain's first token.  Row r
 * attends to the keys anchor[r] sees in the pass (k_pass, v_pass: the pass's
 * [T_pad, Hkv, d] keys and values, as given to spinf_branch_attention), then to the
 * decode rows of its chain from the first token down to itself (k_dec, v_dec:
 * [n_dec, Hkv, d]), with the same softmax: its output equals that of the tokens written
 * into the template and laid out in a pass.  Keys are visited and merged in a fixed
 * order, so a row's output does not depend on the other rows of the call or on where it
 * sits among them.  Rows of one anchor placed next to each other in q_row (a beam's
 * rows) share the reads of their anchor's keys and values.
 *
 * q [n_q, Hq, d] are the queries of decode rows q_row[0..n_q) and o [n_q, Hq, d]
 * receives their outputs (bf16, device, 16-byte aligned).  anchor, parent [n_dec] and
 * q_row [n_q] are device int32 arrays (the decode loop's own state); each row is checked
 * on the device (q_row in range, parents earlier, one anchor per chain, chains of at most
 * 64 tokens, an anchor in the pass whose root path is at most four runs): a row that
 * fails is written as zeros and the plan's error word becomes SPINF_E_DEVICE_CHECK
 * (spinf_device_status).  d_head 64, 128 or 256; 1..8 query heads per kv head;
 * scale <= 0 means 1/sqrt(d).  No window.  Needs the pass uploaded; asynchronous on
 * `stream`.  Errors: SPINF_E_INVALID, SPINF_E_UNSUPPORTED, SPINF_E_CUDA. */
spinf_status spinf_decode_attention(const spinf_plan* plan, int32_t pass, const void* q, const void* k_pass,
                                    const void* v_pass, const void* k_dec, const void* v_dec, int32_t n_dec,
                                    const int32_t* anchor, const int32_t* parent, const int32_t* q_row, int32_t n_q,
                                    void* o, int32_t n_q_heads, int32_t n_kv_heads, int32_t d_head, float scale,
                                    spinf_stream stream);

/* Bytes of device workspace spinf_score_rows needs. */
size_t spinf_score_rows_workspace_bytes(int32_t n_rows, int32_t vocab, int32_t d_model, int32_t w_dtype, int32_t k);

/* Next-token answers at caller-given rows (the decode rows of searched slots): for
 * every row r of hidden [n_rows, d_model] (bf16, device) the full-vocabulary
 * log-sum-exp row_lse[r] and the k tokens (1..16) with the largest logit among the
 * allowed set token_set[r] (device int32 [n_rows], -1 = every token; NULL = every token
 * for all rows), most likely first, ties by lower id, with their z - row_lse (top_tok,
 * top_lp: device [n_rows][k]).  The same kernels as spinf_score_extract, every row a
 * searched row; a set number >= n_sets is read as every token and raises
 * SPINF_E_DEVICE_CHECK.  `plan`: any uploaded plan (its device error word).
 * Asynchronous on `stream`. */
spinf_status spinf_score_rows(const spinf_plan* plan, const void* hidden, int32_t n_rows, const void* w,
                              const float* w_scale, int32_t w_dtype, int32_t d_model, int32_t vocab,
                              const int32_t* token_set, const uint32_t* token_sets, int32_t n_sets, int32_t k,
                              float* row_lse, int32_t* top_tok, float* top_lp, void* workspace, size_t workspace_bytes,
                              spinf_stream stream);

/* Size of the device scratch area behind spinf_score_static: 64 MiB, reserved on
 * every GPU that loads this library, for as long as the process runs. */
#define SPINF_SCORE_STATIC_SCRATCH_BYTES (64u << 20)

/* spinf_score without a workspace argument, for callers that cannot allocate
 * device memory: code running where cudaMalloc is off limits (a host that
 * hands out only pre-planned memory, an allocator hook, a process whose memory
 * is fixed at start-up) or that must not grow its footprint while serving.
 * The pages have no counterpart for this call; it is a deployment convenience.
 *
 * Same arguments, results and errors as spinf_score, minus workspace and
 * workspace_bytes.  The scratch is one file-scope device array of
 * SPINF_SCORE_STATIC_SCRATCH_BYTES per GPU; a pass whose scratch need
 * (spinf_score_workspace_bytes) exceeds it is rejected with SPINF_E_LIMIT
 * before anything is launched.  This call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine); the pass must already have been
 * uploaded with spinf_plan_upload.
 *
 * The first call on a device looks up the device address of its scratch array
 * (cudaGetSymbolAddress, with that device current); make that first call before
 * any stream capture.  The address is kept per device together with the driver
 * context it belongs to: after a cudaDeviceReset (a new context) the next call
 * looks it up again, so that call too should come before any stream capture.  Every call on a device shares the one array and leaves
 * its contents behind; nothing in it has to start at zero (each call writes
 * every byte it later reads).  Calls whose kernels overlap on the GPU -- two
 * streams, or two host threads -- race on the array: order them. */
spinf_status spinf_score_static(const spinf_plan* plan, int32_t pass,
                                const void* hidden, const void* w, const float* w_scale, int32_t w_dtype,
                                int32_t d_model, int32_t vocab,
                                float* row_lse, float* token_lp, spinf_stream stream);

/* Per option lp, p, residual and floor (host, fp64), from each pass's token
 * log-probabilities copied to the host (token_lp_per_pass[p] has G_p floats).
 * Option lp = sum of its token lps in token order; p_o = exp(lp_o - m) /
 * sum_j exp(lp_j - m), m = max_j lp_j; residual = -expm1(logsumexp_j lp_j)
 * ("spinf-serve" news repost, English part: the refund example's response). */
spinf_status spinf_collect(const spinf_plan* plan, const float* const* token_lp_per_pass,
                           const spinf_result* out);

/* Searched-slot answers in question order (input by input, question by question,
 * searched slots only), from each pass's top_tok / top_lp copied to the host:
 * tok [n_extract][extract_k] and lp [n_extract][extract_k] (fp64 copies).  The
 * per-option fields of spinf_collect are absent for a searched slot, and its
 * residual and floor_residual are NaN.  SPINF_E_INVALID for NULL arrays. */
spinf_status spinf_collect_extract(const spinf_plan* plan, const int32_t* const* top_tok_per_pass,
                                   const float* const* top_lp_per_pass, int32_t* tok, double* lp);

/* Wait for `stream`, then report the plan's device error word:
 * SPINF_OK, SPINF_E_DEVICE_TIMEOUT or SPINF_E_DEVICE_CHECK (the word is cleared). */
spinf_status spinf_device_status(const spinf_plan* plan, spinf_stream stream);

/* ---- Around the attention call: the rest of a packed layer (QKV projection with
 * rotary positions, output projection) and the fp8 form of its linears. ---- */

/* Rotary position embedding in place on q [T_pad, Hq, d] and k [T_pad, Hkv, d]
 * (bf16, device): row r's pairs (x[i], x[i + d/2]) turn by pos[r] * theta^(-2i/d),
 * pos[r] being the row's depth on its own root path (spinf_pass_info.pos), so a
 * branch token gets the position it has in its unpacked sequence ("spinf-serve
 * 0.1.1" PyPI, "What it does": branches of one pass, scores equal alone or packed).
 * cos and sin come from a table formed in fp64 on the host and rounded to fp32 (one
 * per pass and (d, theta), built at first use with a synchronous device allocation
 * and kept by the plan); the rotation runs in fp32, bf16 round to nearest.  Pad rows
 * have pos 0 (no change).  Needs the pass uploaded; asynchronous on `stream`.
 * SPINF_E_INVALID for NULL tensors, odd or > 1024 d_head, theta <= 1. */
spinf_status spinf_rope_tree(const spinf_plan* plan, int32_t pass, void* q, void* k, int32_t n_q_heads,
                             int32_t n_kv_heads, int32_t d_head, float theta, spinf_stream stream);

/* y[rows, out] = x[rows, in] . w[out, in]^T on the tensor cores (the output
 * projection of a layer; "one packed forward", man page DESCRIPTION).
 * w_dtype SPINF_DTYPE_BF16: x, w bf16.  SPINF_DTYPE_E4M3 (the static-scale fp8
 * scheme, man page --quant fp8s): x and w are e4m3 codes, w_scale [out] fp32 per
 * output channel, x_scale the static activation scale, and
 * y = (acc * w_scale[o]) * x_scale.  Accumulation fp32, y bf16; all row-major on the
 * device.  Each y element is one fixed-order reduction over `in`, so a row's output
 * does not depend on the other rows.  `plan`: any uploaded plan (its device error
 * word receives a bounded-wait timeout).  in_features a multiple of 8 (16 for e4m3),
 * out_features of 32, pointers 16-byte aligned.  Asynchronous on `stream`. */
spinf_status spinf_linear(const spinf_plan* plan, const void* x, const void* w, const float* w_scale, float x_scale,
                          int32_t w_dtype, void* y, int64_t rows, int64_t in_features, int64_t out_features,
                          spinf_stream stream);

/* The QKV projection of one pass with the rotary embedding fused into its epilogue:
 * [q | k | v] = x[T_pad, d_model] . w[(Hq + 2 Hkv) d, d_model]^T, then q and k turned
 * as spinf_rope_tree does (from the fp32 product, before the one bf16 rounding), and
 * q [T_pad, Hq, d], k, v [T_pad, Hkv, d] written in the layouts spinf_branch_attention
 * reads.  Dtypes and scales as spinf_linear.  d_head in {64, 128, 256}.  Needs the pass
 * uploaded; asynchronous on `stream`. */
spinf_status spinf_qkv_rope(const spinf_plan* plan, int32_t pass, const void* x, const void* w, const float* w_scale,
                            float x_scale, int32_t w_dtype, int32_t d_model, int32_t n_q_heads, int32_t n_kv_heads,
                            int32_t d_head, float theta, void* q, void* k, void* v, spinf_stream stream);

/* e4m3 codes of n bf16 values with a static scale: codes = e4m3(x / x_scale), the
 * division in fp32, round to nearest even, saturating at +-448 (the activation side
 * of the fp8s linears).  n a multiple of 8; x 16-byte, codes 8-byte aligned;
 * x_scale > 0.  Asynchronous on `stream`. */
spinf_status spinf_quantize_static(const void* x, float x_scale, void* codes, int64_t n, spinf_stream stream);

/* Failure-path self-test: enqueue on `stream` a one-thread kernel that waits on a
 * barrier nothing arrives on, with the kernels' bounded wait shortened to `wait_ms`
 * (1..10000); the plan's error word then holds the timeout, which the next
 * spinf_device_status reports as SPINF_E_DEVICE_TIMEOUT (and clears), and the device
 * stays usable.  Nothing faults or hangs.  The pages have no counterpart.
 * SPINF_E_INVALID before any upload or for a bad wait_ms. */
spinf_status spinf_device_selftest(const spinf_plan* plan, int32_t wait_ms, spinf_stream stream);

void spinf_plan_free(spinf_plan* plan);

/* Kernel version, tile configuration and precision: two results are bitwise
 * comparable only when their fingerprints match ("spinf-serve 0.1.1",
 * "What it does": system_fingerprint). */
const char* spinf_fingerprint(void);

const char* spinf_status_string(spinf_status status);

/* Text of the calling thread's last error ("" if none). */
const char* spinf_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPINF_H */
