/*
 * dfl.h -- C ABI of one DFlash speculative-decode step over Q4_1 weights on one GB300 (sm_103a).
 *
 * The step (pages, by title and section):
 *   1. Draft: an 8-row block [last token, mask x 7] conditioned on the target's tapped layer outputs
 *      through the draft's fc projection proposes up to 7 tokens in one pass (model card
 *      "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", spec table and "How it is used"; 1bit engine PR "a Gemma4
 *      pack stops re-reading its weights every token; tools/dflash_acceptance", item 2).
 *   2. Verify: one batched pass of the target over the k drafted rows, every projection one M-row
 *      product, attention over per-layer-width KV planes: sliding and full layers, and KV-shared
 *      layers that read their owner's plane and append nothing (1bit engine PR "npu forward: Gemma4
 *      verifies a draft in one batched pass; KV row width per layer", "What changes").
 *   3. Accept the longest agreeing prefix plus one target token (greedy, first maximum; or sampled
 *      per position), then commit_verify_rows: keep that many rows, pure index arithmetic.
 *
 * Conventions
 *  - Every call returns DFL_OK (0) or a negative DFL_E_* code; dfl_last_error() gives the message.
 *    On any error the state (positions held, planes, draft context) is unchanged.
 *  - Memory: the library never allocates device memory. The caller allocates the three device buffers
 *    sized by dfl_required_bytes() and keeps them alive until dfl_destroy(). Device pointers below
 *    are marked "device"; everything else is host memory.
 *  - Calls enqueue work on the stream given to dfl_init(). Calls with host outputs (tokens, counts,
 *    logits) synchronise that stream before returning, so the outputs are valid on return. Calls
 *    without host outputs return without synchronising.
 *  - Numbers: activations, KV planes and taps are fp32 (the pages' "floats"); weights are Q4_1 or bf16.
 *  - Formats: bf16 = upper half of IEEE binary32. Q4_1 matrix ("container" layout): uint8
 *    [N][K/32][20]; block = fp16 scale d, fp16 minimum m, 16 bytes of 4-bit codes, element i of the
 *    block in byte 4 + i/2 (low nibble for even i); weight w = d*q + m ("Q4_1: 5 bits per weight with
 *    scales and minimums", model card spec table). N = output columns, K = inputs (reduction).
 *  - Not thread-safe: one host thread per context.
 */
#ifndef DFL_H
#define DFL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFL_MAX_LAYERS 64
#define DFL_MAX_TAPS 8
#define DFL_MAX_ROWS 16          /* rows of one verify or prefill chunk (R_max) */

enum {
    DFL_OK = 0,
    DFL_E_INVALID_ARG = -1,      /* bad pointer, size, token id or configuration */
    DFL_E_STATE = -2,            /* call not legal in the current state (e.g. verify while pending) */
    DFL_E_CAPACITY = -3,         /* positions would exceed max_ctx */
    DFL_E_UNSUPPORTED = -4,      /* e.g. k > DFL_MAX_ROWS, a shape the kernels do not take */
    DFL_E_CUDA = -5,             /* a CUDA call failed; the message names it */
    DFL_E_TIMEOUT = -6           /* a bounded device wait gave up (about 1 s); reported by the next call
                                    that reads the device state, with the state of the last good call */
};

enum { DFL_SLIDING = 0, DFL_FULL = 1 };

/* Model and capacity. Layer l is KV-shared when kv_owner[l] != l: it reads the plane of layer
 * kv_owner[l] (the last non-shared layer of the same attention type) and appends nothing. */
typedef struct dfl_config {
    /* target */
    int32_t n_layers, hidden, vocab, n_heads, head_dim;
    int32_t window;                        /* sliding window: keys p-window+1..p visible to position p */
    int32_t ple_dim;                       /* per-layer-embedding width; 0 = none (and no layer scalar) */
    int32_t layer_type[DFL_MAX_LAYERS];    /* DFL_SLIDING / DFL_FULL */
    int32_t kv_heads[DFL_MAX_LAYERS];
    int32_t kv_owner[DFL_MAX_LAYERS];
    int32_t ffn[DFL_MAX_LAYERS];
    float rope_base_sliding, rope_base_full, eps, emb_scale;
    /* draft (hidden width = target hidden) */
    int32_t d_layers, d_ffn, d_heads, d_kv_heads, d_head_dim;
    int32_t d_window;                      /* context keys visible to a block; 0 = all */
    int32_t block;                         /* rows of a draft block (proposals = block - 1) */
    int32_t n_taps, mask_token;
    int32_t taps[DFL_MAX_TAPS];            /* target layers whose outputs feed fc, ascending */
    float d_rope_base, d_eps, d_emb_scale;
    /* capacity */
    int32_t max_ctx;                       /* positions the KV arena holds */
    int32_t prefill_rows;                  /* 0, or 128..8192 (a multiple of 16): dfl_prefill takes up to
                                              this many prompt rows in one pass whose products run on the
                                              tcgen05 tensor cores (the buffers of such a pass, and sliding
                                              rings of window + prefill_rows - 1 slots, are sized in) */
} dfl_config;

typedef struct dfl_sizes {
    uint64_t weights_bytes;                /* packed weight image, tables */
    uint64_t state_bytes;                  /* KV planes, draft context, taps, device counters */
    uint64_t workspace_bytes;              /* activations and reduction scratch of one pass */
} dfl_sizes;

typedef struct dfl_buffers {
    void *weights;                         /* device, >= weights_bytes, 256-byte aligned */
    void *state;                           /* device, >= state_bytes, 256-byte aligned */
    void *workspace;                       /* device, >= workspace_bytes, 256-byte aligned */
} dfl_buffers;

/* Sampling: temperature > 0 samples every verified position with the uniform
 * U(seed, position) = top 53 bits of SplitMix64(seed XOR position * 0x9E3779B97F4A7C15) * 2^-53,
 * and picks the smallest token whose running sum of exp((l - max)/T) exceeds U * sum.
 * A NULL dfl_sampling, or temperature <= 0, means greedy (first maximum). */
typedef struct dfl_sampling {
    float temperature;
    uint64_t seed;
} dfl_sampling;

typedef struct dfl_ctx dfl_ctx;

/* Sizes of the three device buffers for a configuration. Fails with DFL_E_INVALID_ARG or
 * DFL_E_UNSUPPORTED on a configuration the library does not take (it states which field). */
int dfl_required_bytes(const dfl_config *cfg, dfl_sizes *out);

/* Create a context over caller-owned device buffers (sizes from dfl_required_bytes) and a CUDA
 * stream (cudaStream_t, may be NULL for the legacy stream). Positions held start at 0. Every tensor
 * must then be given once with dfl_load_tensor before the first pass. The context does not own the
 * buffers or the stream. */
int dfl_init(const dfl_config *cfg, const dfl_buffers *buf, void *cuda_stream, dfl_ctx **out);

/* Load one tensor from DEVICE memory in its container format; the library packs it into its own
 * layout in the weights buffer (Q4_1 matrices into a tile-major image of the same bytes per weight).
 * Names: "emb" bf16 [vocab][hidden]; "head" bf16 [vocab][hidden]; "final_norm" bf16 [hidden];
 * "ple_table" bf16 [vocab][n_layers*ple_dim]; per target layer l, "t<l>.": attn_norm, q_norm,
 * k_norm (owners), post_attn_norm, pre_ffn_norm, post_ffn_norm, ple_norm (bf16), lambda (bf16 [1]),
 * wqkv (owners: q|k|v) or wq (shared), wo, wgu (gate|up), wd, wple_g, wple_p (Q4_1);
 * draft: "d.fc" bf16 [hidden][n_taps*hidden], "d.hidden_norm", "d.final_norm", and per draft
 * layer "d<l>.": attn_norm, q_norm, k_norm, ffn_norm, wqkv, wo, wgu, wd.
 * `bytes` must equal the tensor's container size. The source may be freed once the stream has
 * passed this call (it is read by kernels enqueued here). */
int dfl_load_tensor(dfl_ctx *ctx, const char *name, const void *dev_src, size_t bytes);

/* Prefill (extend the context; 1bit engine PR "npu forward: Gemma4 verifies a draft in one batched
 * pass; KV row width per layer", "What changes" item 1, extend_context): run the n tokens at positions
 * held..held+n-1 in passes, commit them, bring the draft context up to date,
 * and write the target's token for the next position to *next_tok (greedy or sampled). The output
 * head runs on the last prompt row only: only that row's token is needed. Passes: with prefill_rows > 0,
 * min(prefill_rows, remaining) rows while 128 or more remain (products on tcgen05), then passes of at
 * most DFL_MAX_ROWS rows; with prefill_rows = 0, passes of at most DFL_MAX_ROWS rows. Fails with
 * DFL_E_CAPACITY if held + n exceeds max_ctx; on any error positions held stay as they were. An error
 * after the first pass was enqueued (DFL_E_TIMEOUT, DFL_E_CUDA) on a context that held positions
 * leaves it refusing passes and snapshots with DFL_E_STATE until dfl_restore succeeds: the passes that
 * ran may have overwritten sliding-ring and draft-context slots those positions still need. */
int dfl_prefill(dfl_ctx *ctx, const int32_t *tokens, int n, const dfl_sampling *s, int32_t *next_tok);

/* Draft block (model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", "How it is used"; 1bit engine PR "a
 * Gemma4 pack stops re-reading its weights every token; tools/dflash_acceptance", item 2) at positions
 * held..held+block-1 for rows [last_tok, mask x (block-1)]: first makes the committed rows not yet in
 * the draft context into context (fc of their taps, then each draft layer's key and value), then runs
 * the block. Proposals (block-1 tokens for positions held+1..) are kept on the device for
 * dfl_verify_block(rows = NULL) and copied to `proposals` when it is not NULL (which synchronises; with
 * NULL the call does not synchronise, and a device error surfaces at the next synchronising call). */
int dfl_draft_block(dfl_ctx *ctx, int32_t last_tok, int32_t *proposals);

/* Batched verify (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass; KV row
 * width per layer", "What changes": every projection one M-row product, a KV-shared layer reads its
 * owner's plane and appends nothing; acceptance: model card "How it is used") of k rows at positions
 * held..held+k-1. rows = [last token, proposal 1, .., proposal k-1]; rows == NULL takes last_tok of the
 * last draft block and its k-1 first proposals. Writes the target's token for positions
 * held+1..held+k to target_tok[0..k-1] (if not NULL) and the accepted length a (longest prefix with
 * proposal i == target token i-1) to *accepted (if not NULL). The tokens the pass emits are
 * target_tok[0..a] (the accepted proposals equal the target's tokens before them, plus the target's
 * token after the last one). The rows stay pending until dfl_commit_verify_rows / dfl_commit_accepted.
 * k in 1..DFL_MAX_ROWS. */
int dfl_verify_block(dfl_ctx *ctx, const int32_t *rows, int k, const dfl_sampling *s,
                     int32_t *target_tok, int32_t *accepted);

/* commit_verify_rows (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass",
 * "What changes" item 1 and "Proof": 3 held, commit_verify_rows(2), 5 held): keep the first `keep` rows
 * of the pending verify (0 <= keep <= k); positions held become held + keep. Pure index arithmetic: no
 * data moves; later rows are overwritten by the next pass. keep = DFL_KEEP_ACCEPTED keeps accepted + 1
 * rows (the accepted proposals and the row of the last token) as counted by the last verify. */
#define DFL_KEEP_ACCEPTED (-1)
int dfl_commit_verify_rows(dfl_ctx *ctx, int keep);
/* The acceptance step's commit (model card "How it is used": the longest agreeing prefix plus one
 * target token are kept): keep min(accepted + 1, max_keep) rows of the pending verify, where max_keep
 * caps the tokens a caller still wants (a token budget), and write that count to *kept (if not NULL).
 * The tokens the kept rows emit are target_tok[0..*kept-1] of the verify. With stop_token >= 0, a kept
 * row whose token is the stop token ends the count there: that token is emitted, but no row for it is
 * ever committed (single-turn serving, FastFlowLM PR #899 "gemma4e-dflash-flash", "Changes": no KV row
 * for the stop token); *stopped (if not NULL) is then 1, else 0. */
int dfl_commit_accepted(dfl_ctx *ctx, int max_keep, int32_t stop_token, int32_t *kept, int32_t *stopped);

/* Snapshot (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass", "What changes"
 * item 1: snapshot and restore cut each plane at its own layer's width; a KV-shared layer's plane stays
 * empty) of the committed state (positions held, every owner plane, the draft context, the taps of
 * committed rows not yet in the draft context) into a DEVICE buffer of at least dfl_snapshot_bytes()
 * bytes; restore replaces the state with a snapshot taken from a context with the same configuration.
 * Both need the committed state (no pending verify). KV-shared layers have no plane and contribute
 * nothing. A snapshot taken once after a pinned prefix may be restored any number of times (FastFlowLM
 * PR #899 "gemma4e-dflash-flash", "Changes": the pinned prefix must not be overwritten by a request). */
int64_t dfl_snapshot_bytes(const dfl_ctx *ctx);
int dfl_snapshot(dfl_ctx *ctx, void *dev_dst, size_t bytes);
int dfl_restore(dfl_ctx *ctx, const void *dev_src, size_t bytes);

/* Per-layer KV row width in floats per position (1bit engine PR "npu forward: Gemma4 verifies a draft
 * in one batched pass", "What changes" item 1, kv_widths(): 2 x 256 on E4B's sliding layers, 2 x 512 on
 * its full layers): 2 * kv_heads * head_dim for a layer with its own plane, 0 for a KV-shared layer.
 * out: n_layers entries. */
int dfl_kv_widths(const dfl_ctx *ctx, int32_t *out);

/* Positions held (committed), counted over owner planes only (same PR, "What changes" item 1: the
 * positions-held count ignores shared layers). -1 on a NULL context. */
int64_t dfl_positions_held(const dfl_ctx *ctx);

/* Options. DFL_OPT_KEEP_LOGITS = 1 makes verify and draft passes also store their fp32 logits
 * (otherwise only the fused argmax runs); DFL_OPT_GRAPHS = 0 launches kernels one by one instead of
 * replaying captured CUDA graphs; DFL_OPT_STOP_LAYER = l >= 0 (inspection only) makes target passes
 * stop after layer l, without the head, so dfl_debug_read shows that layer's intermediates; -1 = off;
 * DFL_OPT_PROFILE = 1 times the kernel launches of every pass on the device (read with
 * dfl_profile_read; setting the option clears the totals; each profiled pass synchronises once, to read
 * its time stamps); DFL_OPT_ATTN_CLUSTER = 16 (default), 8 or 4
 * caps the number of CTAs over which attention spreads one pair of query heads (the largest size up to
 * the cap whose clusters all fit on the device at once is taken; sizes differ in the order in which
 * the partial softmax states are added, so logits may differ in the last bits); other values are
 * DFL_E_INVALID_ARG. Changing it drops the captured graphs. */
enum { DFL_OPT_KEEP_LOGITS = 1, DFL_OPT_GRAPHS = 2, DFL_OPT_STOP_LAYER = 3, DFL_OPT_PROFILE = 4,
       DFL_OPT_ATTN_CLUSTER = 5, DFL_OPT_TEST_STALL = 6, DFL_OPT_FUSE_STEPS = 7, DFL_OPT_PLE_SPLIT = 8 };
/* DFL_OPT_PLE_SPLIT = 1 runs the per-layer-embedding tail's gate and projection (PR-batched "What
 * changes": gate = silu(x Wg) times the layer's per-layer input, then its projection) as two products
 * (0, the default, runs them as one launch on a cluster of ple_dim / 16 CTAs when the pass has at most
 * 16 rows and ple_dim is a multiple of 16 up to 256). Both give results within the parity tolerance of
 * each other. Changing it drops the captured graphs. */
/* DFL_OPT_FUSE_STEPS = 1 runs the row steps (residual, norms, layer scalar, taps) and the q/k steps
 * (norm, rotation, KV store) on the last CTAs of the product that feeds them instead of as separate
 * kernels (0, the default). Both give results within the parity tolerance of each other (the sums are
 * taken in different orders); on the E4B-shaped pair the separate kernels are faster. Changing it drops
 * the captured graphs. */
/* DFL_OPT_TEST_STALL = 1 (tests of the error path only): the Q4_1 products of the following passes
 * issue no copies, so the first one's bounded waits give up after about a second and the call that reads
 * the device state returns DFL_E_TIMEOUT with the state unchanged; set it back to 0 and the context
 * works as before. */
int dfl_set_option(dfl_ctx *ctx, int option, int value);

/* Copy the fp32 logits of the last pass (rows x vocab, row-major) to host memory. which = 0: the
 * last verify block (rows <= its k) or, after dfl_prefill, the last prompt row (rows = 1); which = 1:
 * the last draft block (rows 1..block-1, rows <= block-1). Needs DFL_OPT_KEEP_LOGITS. */
int dfl_read_logits(dfl_ctx *ctx, int which, float *host_dst, int rows);

/* Copy the fp32 taps of positions pos0..pos0+rows-1 (n_taps*hidden each) to host memory. */
int dfl_read_taps(dfl_ctx *ctx, int pos0, int rows, float *host_dst);

/* Draft-only context: make `rows` rows of given taps (DEVICE fp32 [rows][n_taps*hidden]) context at
 * positions held..held+rows-1 and advance positions held, without running the target. A context used
 * this way refuses dfl_verify_block and dfl_prefill (DFL_E_STATE). */
int dfl_draft_append_taps(dfl_ctx *ctx, const void *dev_taps, int rows);

/* Inspection: copy the first `bytes` of an internal buffer of the last pass to host memory. Names:
 * "x" [16][hidden] residual rows, "y" [16][hidden] last projection output, "qkv" [16][width],
 * "q" [16][heads*head_dim] (normed, rotated), "x_d" [16][hidden] draft residual rows; "k<l>" and "v<l>"
 * the key and value plane of target layer l, [slots][kv_heads][head_dim] with position p in slot p
 * (full layers) or p mod (window + 15) (sliding layers); all fp32. A KV-shared layer has no plane
 * (DFL_E_INVALID_ARG). */
int dfl_debug_read(dfl_ctx *ctx, const char *name, void *host_dst, size_t bytes);

/* Planted drafts (measurement workloads that control acceptance): after dfl_draft_block, replace its
 * proposals on the device with dev_table[held+1 .. held+block-1], a DEVICE int32 table indexed by
 * absolute position with at least held+block entries. The draft block itself has run. */
int dfl_plant_proposals(dfl_ctx *ctx, const int32_t *dev_table, int table_len);

/* Kernels this context has launched so far (every launch counted once). */
int64_t dfl_launch_count(const dfl_ctx *ctx);

/* Totals of the launches profiled while DFL_OPT_PROFILE was on, per class: 0 = Q4_1 products,
 * 1 = bf16 products (fc), 2 = the bf16 head with its fused argmax, 3 = attention, 4 = q/k norm,
 * rotation and KV store, 5 = the row kernels (residual and norms, taps), embedding and sampling (the
 * small state and copy kernels are not timed). A launch's time is its in-pass duration on the device
 * clock: from the earliest of its CTAs past its dependency wait to the latest of its CTAs done, so the
 * overlap of consecutive launches (programmatic dependent launch) is kept and the durations of a
 * pass's launches add up to at most the pass. *ms = their sum; *bytes = the launches' algorithmic
 * bytes for classes 0-2 (weights at 0.625 B (Q4_1) or 2 B (bf16) per weight, fp32 activations in and
 * products out), 0 for the others. Error DFL_E_INVALID_ARG for a class outside 0..5. Synchronises the
 * stream. */
int dfl_profile_read(dfl_ctx *ctx, int cls, int64_t *launches, double *ms, double *bytes);

const char *dfl_last_error(const dfl_ctx *ctx);
void dfl_destroy(dfl_ctx *ctx);

/* ---- the Q4_1 product on its own (used for the isolated GEMM measurements) ----------------------- */

/* Bytes of the packed tile image of a K x N Q4_1 matrix (K padded up to a multiple of 64). */
int64_t dfl_q41_image_bytes(int K, int N);
/* Pack a container-layout Q4_1 matrix (DEVICE) into the tile image (DEVICE). */
int dfl_q41_pack(const void *dev_src, int K, int N, void *dev_image, void *cuda_stream);
/* Bytes of an activation operand buffer for up to 16 rows of K inputs (K % 16 == 0). */
int64_t dfl_act_bytes(int M, int K);
/* Pack fp32 rows x (DEVICE [M][K]) into an activation operand buffer (DEVICE, dfl_act_bytes): bf16
 * hi + lo fragments in the order the tensor cores consume them, and per-16-input sums. */
int dfl_act_pack(const float *dev_x, int M, int K, void *dev_act, void *cuda_stream);
/* Scratch bytes dfl_q41_gemm needs for K, N, M. */
int64_t dfl_q41_gemm_scratch_bytes(int K, int N, int M);
/* y[m][n] = sum_k x[m][k] * w[k][n] (fp32), x given as an activation operand buffer (DEVICE, from
 * dfl_act_pack), y fp32 DEVICE [M][N], from the tile image; M in 1..16; N a multiple of 32. The
 * scratch (DEVICE, 256-byte aligned, >= dfl_q41_gemm_scratch_bytes) holds an error word (its first 4
 * bytes), arrival counters and partial sums; it must be zeroed once before the first call (each call
 * leaves the counters zero). Calls on one scratch must not overlap on the GPU. A row's result does not
 * depend on M. The call only enqueues; a bounded wait that gave up sets the error word (read it with
 * dfl_q41_gemm_status) and leaves y undefined. */
int dfl_q41_gemm(const void *dev_image, int K, int N, const void *act, int M, float *dev_y,
                 void *dev_scratch, size_t scratch_bytes, void *cuda_stream);
/* Status of the products enqueued on a scratch so far: synchronises the stream, returns DFL_OK, or
 * DFL_E_TIMEOUT (and clears the error word) when a bounded wait of one of them gave up. */
int dfl_q41_gemm_status(const void *dev_scratch, void *cuda_stream);

/* ---- the Q4_1 product at many rows (prompt ingest) on the tcgen05 tensor cores -------------------- */

/* Scratch bytes dfl_q41_gemm_tc needs for K, N, M (the weights expanded to bf16 hi + lo, N x Kp x 4
 * bytes, and the rows split the same way, M x Kp x 4 bytes, Kp = K rounded up to 64, plus a 1 KiB
 * header), or -1 for a shape it does not take (K and N multiples of 32 as for the tile image, M >= 1). */
int64_t dfl_q41_gemm_tc_scratch_bytes(int K, int N, int M);
/* y[m][n] = sum_k x[m][k] * w[k][n] for a Q4_1 tile image (DEVICE, dfl_q41_pack), fp32 rows x (DEVICE
 * [M][K], row-major) and fp32 y (DEVICE [M][N], row-major). 1bit engine PR "npu forward: Gemma4
 * verifies a draft in one batched pass", "What changes" item 1: a prompt goes through the layer
 * products in chunks of rows; this is that product for chunks of hundreds of rows, where it is a
 * dense contraction. w = d q + m is formed in fp32 and split into bf16 hi + lo, x likewise; the
 * tensor cores add hi*hi + hi*lo + lo*hi in fp32, so y carries about the error of an fp32 dot
 * product (it is not bit-identical to dfl_q41_gemm's). The scratch (DEVICE, 1024-byte aligned, >=
 * dfl_q41_gemm_tc_scratch_bytes) starts with the error word of dfl_q41_gemm_status, which must be
 * zero before the first call and reports (DFL_E_TIMEOUT) a bounded device wait that gave up, leaving
 * y undefined. Calls on one scratch must not overlap on the GPU. The call only enqueues three kernels
 * on the stream (weight expansion, row split, product). DFL_E_INVALID_ARG for a shape, pointer, size
 * or alignment it rejects; DFL_E_CUDA when the tensor-map encoder is unavailable or a launch fails. */
int dfl_q41_gemm_tc(const void *dev_image, int K, int N, const float *dev_x, int M, float *dev_y,
                    void *dev_scratch, size_t scratch_bytes, void *cuda_stream);

/* ---- the bf16 head on its own (the isolated sweep's bf16 2560 x 262144 comparison shape) ---------- */

/* Bytes of the packed tile image of a bf16 K x N matrix (K a multiple of 64, N of 16). */
int64_t dfl_bf16_image_bytes(int K, int N);
/* Pack a bf16 matrix [N][K] (DEVICE, row n = output n) into the tile image (DEVICE). */
int dfl_bf16_pack(const void *dev_src, int K, int N, void *dev_image, void *cuda_stream);
/* Scratch bytes dfl_bf16_head_argmax needs. */
int64_t dfl_bf16_head_scratch_bytes(int K, int N, int M);
/* The head product of the step with its fused argmax (model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2",
 * "How it is used": greedy proposals and target tokens are the first maximum of the logits):
 * argmax[m] = the first n maximising sum_k x[m][k] * w[k][n] (DEVICE int32 [M]); logits (DEVICE fp32
 * [M][N], nullable) receives the products themselves. Activations as for dfl_q41_gemm; the scratch
 * (DEVICE, 256-byte aligned, zeroed once before the first call; each call leaves it reusable) must not
 * be shared by calls that overlap on the GPU. */
int dfl_bf16_head_argmax(const void *dev_image, int K, int N, const void *dev_act, int M, int32_t *dev_argmax,
                         float *dev_logits, void *dev_scratch, size_t scratch_bytes, void *cuda_stream);

/* The same product for callers that cannot allocate device memory per call and have no scratch
 * buffer of their own to pass: code that must keep every device allocation out of its call path (a
 * fixed device-memory budget reserved up front), or hosts whose plug-in interface hands over only the
 * input and output pointers. Nothing in the DFlash method corresponds to this entry point; it is a
 * packaging of dfl_q41_gemm.
 * Scratch: one array of dfl_q41_gemm_noalloc_max_scratch() bytes (4 MiB) in the library's static device
 * memory. The first call on a device looks up that device's copy of the array (cudaGetSymbolAddress,
 * with the device current) and caches its address; make that first call outside any stream capture.
 * The cached address belongs to the device's context of that moment: after cudaDeviceReset (or any
 * other teardown of the primary context) call dfl_q41_gemm_noalloc_reset before the next product.
 * No call allocates or frees memory. Every call on a device uses the same array and leaves the last
 * call's contents in it: the arrival counters at its start must be zero, which the zero-initialised
 * array gives and every completed call restores; calls that overlap on the GPU race on it.
 * Errors: DFL_E_INVALID_ARG for the shapes or pointers dfl_q41_gemm rejects; DFL_E_CAPACITY when
 * dfl_q41_gemm_scratch_bytes(K, N, M) exceeds the array; DFL_E_CUDA when the address lookup or the
 * launch fails. Arguments as for dfl_q41_gemm. */
int dfl_q41_gemm_noalloc(const void *dev_image, int K, int N, const void *dev_act, int M, float *dev_y,
                         void *cuda_stream);
/* Bytes of the static scratch array behind dfl_q41_gemm_noalloc. */
int64_t dfl_q41_gemm_noalloc_max_scratch(void);
/* dfl_q41_gemm_status for the static array of the current device. */
int dfl_q41_gemm_noalloc_status(void *cuda_stream);
/* Look the current device's array up again and zero all of it (cudaMemsetAsync on the given stream):
 * after a context teardown, or to start from a known state. Must not overlap a product on the GPU. */
int dfl_q41_gemm_noalloc_reset(void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* DFL_H */
