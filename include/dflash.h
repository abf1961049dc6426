/*
 * dflash.h -- C ABI of the GB300 (sm_103a) block-diffusion drafting library.
 *
 * The library computes one DFlash-style draft step and its greedy
 * verification on one GPU:
 *
 *   dflash_ctx_fuse      hidden states tapped at several target layers are
 *                        fused by a linear layer (+ RMSNorm) into one dense
 *                        context feature.  ("DFlash: how block diffusion
 *                        boosts NVIDIA Blackwell throughput", section "Block
 *                        diffusion architecture", feature-injection item.)
 *   dflash_kv_append     the feature is projected through every draft layer's
 *                        own K/V weights and written into the paged draft KV
 *                        cache, where it persists across iterations.  (Same
 *                        page and section, KV-cache item.)
 *   dflash_draft_block   one non-causal pass of the drafter over
 *                        [anchor, mask x (B-1)]: every block row attends to
 *                        all context keys and all block keys; shared LM head;
 *                        argmax gives B-1 draft tokens.  (Same page, section
 *                        "Block diffusion architecture": parallel block
 *                        denoising in one pass; "DFlash-2: z-lab boosts
 *                        speculative decoding throughput...", section
 *                        "DFlash-2 mechanisms": non-causal drafter, and
 *                        "Architecture upgrade details": the optional local
 *                        convolution between attention and MLP.)  It can also
 *                        append pending context rows in the same weight pass.
 *   dflash_verify_greedy temperature-0 verification: accept the longest prefix
 *                        of drafts equal to the target's argmax, then the
 *                        target's own token; compacts the emitted tokens and
 *                        advances lengths and the anchor.  ("NVIDIA tests
 *                        DFlash to cut LLM inference bottlenecks", section
 *                        "DFlash moves drafting to parallel compute": the
 *                        target keeps the final verification.)
 *
 * Conventions for every call
 *   - Tensors are device pointers to dense row-major arrays.  "bf16" means
 *     bfloat16 bit patterns (uint16_t), round-to-nearest-even.
 *   - The caller owns all memory (weights, KV pools, page tables, workspace,
 *     outputs).  Compute calls allocate nothing; dflash_model_create allocates
 *     only the small per-model descriptor block it frees in destroy.
 *   - All compute calls are asynchronous on `stream` (a cudaStream_t; NULL =
 *     the legacy default stream) and never synchronise, except
 *     dflash_get_status.
 *   - Return value 0 = OK, negative = error (DFLASH_ERR_*); nothing is launched
 *     when a call returns an argument error.  Errors found on the device (a
 *     page-table entry out of range, a wait that timed out) are recorded in the
 *     workspace's status word and read with dflash_get_status.
 *   - A workspace must not be used by two calls that may run concurrently.
 *     dflash_workspace_init must run once on a fresh workspace (and again
 *     after a call reported an error) before it is used.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_OK 0
#define DFLASH_ERR_INVALID_ARG (-1) /* null pointer, misalignment, size out of range */
#define DFLASH_ERR_UNSUPPORTED (-2) /* shape the kernels do not implement        */
#define DFLASH_ERR_CAPACITY (-3)    /* workspace / page table / cache too small    */
#define DFLASH_ERR_CUDA (-4)        /* a CUDA runtime/driver call failed           */
#define DFLASH_ERR_TIMEOUT (-5)     /* a bounded device wait gave up               */
#define DFLASH_ERR_NO_DEVICE (-6)   /* no sm_103 device or driver entry point      */

typedef struct dflash_model_s* dflash_model;

/* Shape of a decoder-layer stack: the drafter, or (for the end-to-end loop)
 * the target.  Supported: hidden % 128 == 0, hidden <= 8192, head_dim in {64, 128},
 * n_q_heads % n_kv_heads == 0 with group n_q_heads/n_kv_heads in {1,2,4,8},
 * (n_q_heads + 2 n_kv_heads) * head_dim % 128 == 0, mlp % 64 == 0,
 * vocab % 128 == 0, block in 1..32 (drafter), conv_width in {0,1,3,5,7},
 * page_size == 16. */
typedef struct {
  int32_t n_layers;
  int32_t hidden;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t mlp;
  int32_t vocab;
  int32_t block;      /* drafter block size B (anchor + B-1 masks); 0 for a target */
  int32_t n_taps;     /* drafter: number of tapped target layers fused by fc       */
  int32_t conv_width; /* DFlash-2 depthwise conv over block positions, 0 = off     */
  int32_t qk_norm;    /* 1 = per-head RMSNorm on q and k before RoPE               */
  int32_t fc_norm;    /* 1 = RMSNorm after the fuse linear                         */
  int32_t page_size;  /* KV page size in positions (16)                            */
  float rms_eps;
  float rope_base;
  /* K/V cache terms: 1 = K and V in bf16; 2 = each stored as two bf16 planes
   * hi = bf16(v), lo = bf16(v - hi) (about 16 significant bits; the attention
   * multiplies both into one fp32 accumulator).  2 is for a target model only:
   * its logits at 8 layers and H = 4096 stay within 0.05 of exact arithmetic
   * only with the two-term cache.  0 is read as 1. */
  int32_t kv_terms;
} dflash_config;

/* Device pointers, all bf16, stacked over layers where marked [L].
 * Rows of a linear weight are output features: y = x W^T.
 * Base pointers must be 16-byte aligned. */
typedef struct {
  const void* embed;      /* [vocab][hidden]      token embedding (shared)      */
  const void* lm_head;    /* [vocab][hidden]      LM head (shared)              */
  const void* final_norm; /* [hidden]                                           */
  const void* in_norm;    /* [L][hidden]          pre-attention RMSNorm gain    */
  const void* wqkv;       /* [L][(hq+2hkv)*d][hidden]  q rows, k rows, v rows   */
  const void* q_norm;     /* [L][d]               (qk_norm)                     */
  const void* k_norm;     /* [L][d]               (qk_norm)                     */
  const void* wo;         /* [L][hidden][hq*d]                                  */
  const void* post_norm;  /* [L][hidden]          pre-MLP RMSNorm gain          */
  const void* w_gate_up;  /* [L][2*mlp][hidden]   gate rows [0,mlp), up rows    */
  const void* w_down;     /* [L][hidden][mlp]                                   */
  const void* conv;       /* [L][hidden][conv_width] or NULL                    */
  const void* fc;         /* [hidden][n_taps*hidden]  drafter fuse linear       */
  const void* fc_norm;    /* [hidden]                                           */
  const void* mask_embed; /* [hidden]             drafter mask-token input      */
} dflash_weights;

/* A paged KV cache (the drafter's context cache, or the target's cache).
 * pool: bf16 [n_layers][n_pages][2*kv_terms][n_kv_heads][page_size][head_dim]
 *       (plane 0 = K after k-norm and RoPE, plane 1 = V; with kv_terms = 2,
 *       planes 2 and 3 hold the low terms of K and V);
 * page_table: int32 [n_rows][max_pages], entry = physical page index; row r
 * belongs to request r (n_rows = the requests the cache can hold).
 * Logical position p of request r lives in page page_table[r][p / page_size]
 * at slot p % page_size.  Pages may be in any physical order.  Request
 * indices read from device arrays (row_req, pending_req) outside
 * [0, n_rows), and page ids outside [0, n_pages), are recorded as
 * DFLASH_ERR_CAPACITY in the workspace status word and the row is skipped. */
typedef struct {
  void* pool;
  const int32_t* page_table;
  int32_t n_pages;
  int32_t max_pages;
  int32_t n_rows;
  /* 0: the pool holds bf16 K/V.  1 (drafter context caches): the pool holds
   * E4M3 codes, uint8 [n_layers][n_pages][2][n_kv_heads][page_size][head_dim],
   * and `scales` fp32 [n_layers][n_pages][2][n_kv_heads][page_size] one scale
   * per (position, head) of K and of V: value = decode(code) * scale, with
   * scale = amax / 448 of the vector's bf16 values (1 for a zero vector) and
   * codes rounded to nearest, ties to even, saturating at +-448 ("DFlash-2:
   * z-lab boosts speculative decoding throughput...", section on the
   * precision cost: an 8-bit KV cache against a 16-bit one). */
  int32_t dtype;
  float* scales;
} dflash_kv;

/* ------------------------------------------------------------------ model */

/* Builds the TMA descriptors for the weights and checks the shape.  Copies
 * *cfg and *w; the weight memory must outlive the model.  Requires a current
 * CUDA device of compute capability 10.3. */
int dflash_model_create(const dflash_config* cfg, const dflash_weights* w, dflash_model* out);
int dflash_model_destroy(dflash_model m);

/* Workspace bytes for calls with up to `max_block_rows` block (or target)
 * rows, `max_ctx_rows` context rows and `max_batch` requests whose context
 * is at most `max_ctx_len` positions.  The workspace must be 256-byte aligned. */
size_t dflash_workspace_bytes(dflash_model m, int32_t max_block_rows, int32_t max_ctx_rows,
                              int32_t max_batch, int32_t max_ctx_len);
/* Zeroes the workspace header (status word and split counters). */
int dflash_workspace_init(void* ws, size_t ws_bytes, void* stream);
/* Synchronises `stream`, copies the workspace status word to the host and
 * returns it (0 = no device-side error) through *status; *site gets the
 * raising kernel's site id (may be NULL). */
int dflash_get_status(const void* ws, int32_t* status, int32_t* site, void* stream);
const char* dflash_strerror(int code);
/* Number of kernels this library has launched from the host in this process
 * (launches replayed from a captured CUDA graph are not counted). */
uint64_t dflash_kernel_launches(void);
/* CUDA error code of the last DFLASH_ERR_CUDA on this thread (0 if none). */
int dflash_last_cuda_error(void);

/* ------------------------------------------------------------- hot path */

/* c = RMSNorm_fc(taps W_fc^T) for T rows.
 * taps: bf16 [T][n_taps*hidden] (tapped hidden states, listed-layer order);
 * ctx:  bf16 [T][hidden] output.  1 <= T <= max_ctx_rows of the workspace. */
int dflash_ctx_fuse(dflash_model m, const void* taps, int32_t T, void* ctx, void* ws,
                    size_t ws_bytes, void* stream);

/* For every layer l: K = RoPE(knorm(W_k^l c_t), pos_t), V = W_v^l c_t, stored
 * at logical position row_pos[t] of request row_req[t].  Rows with
 * row_pos[t] < 0 are skipped.  ctx: bf16 [T][hidden].  m must be a drafter
 * (DFLASH_ERR_INVALID_ARG for a target model).  A row_req[t] outside
 * [0, kv->n_rows) is recorded as DFLASH_ERR_CAPACITY in the status word and
 * its row is skipped. */
int dflash_kv_append(dflash_model m, const void* ctx, const int32_t* row_req,
                     const int32_t* row_pos, int32_t T, const dflash_kv* kv, void* ws,
                     size_t ws_bytes, void* stream);

/* dflash_ctx_fuse for callers that cannot allocate device memory (for
 * example code running while another framework owns or has reserved the whole
 * device memory pool, or that may not grow its footprint after start-up).  The
 * pages describe no such call; it exists for deployment only.
 * Same inputs and output as dflash_ctx_fuse, no workspace argument: the
 * scratch is a fixed 4 MiB array inside the library, held by every GPU that
 * loads the library until the process exits.  Needs 64 KiB + T*hidden*4 bytes
 * of it, so T <= (4 MiB - 64 KiB) / (hidden*4): 252 rows at hidden 4096,
 * 2016 at hidden 512.  A larger T, like any other bad argument, is rejected
 * (DFLASH_ERR_CAPACITY) before the array is touched or anything is launched.
 * The first call on a device looks up the array's device address; make that
 * first call before any stream capture.  The address is kept for the device's
 * primary context: after that context is destroyed (cudaDeviceReset) it is
 * stale, and this call must not be used again in the process.  All calls
 * share the array (the header is cleared at the start of each call that
 * launches), so calls that may overlap on the GPU (different streams, or
 * devices sharing a context) race.  Device-side status is not reported back. */
int dflash_ctx_fuse_noalloc(dflash_model m, const void* taps, int32_t T, void* ctx,
                            void* stream);

/* One drafter pass for `batch` requests (batch <= kv->n_rows, else
 * DFLASH_ERR_CAPACITY before any launch).  Request r's anchor token
 * anchor[r] sits at position L_r = anchor_pos[r]; block position i at L_r+i;
 * block rows attend to context positions [0, L_r) of the cache and to all B
 * block positions.  If T > 0, the T pending context rows (pending_ctx bf16
 * [T][hidden], pending_req, pending_pos, as in dflash_kv_append) are
 * projected in the same weight pass and written to the cache before
 * attention reads it.
 * Outputs: draft int32 [batch][B-1] (argmax of rows 1..B-1, lowest index on
 * ties); optional logits fp32 [batch*B][vocab] and hidden fp32
 * [batch*B][hidden] (final residual stream before the final norm) for
 * checking; pass NULL to skip them.
 * With an E4M3 cache (kv->dtype 1) the pending rows are stored as codes and
 * scales, and attention decodes the context keys exactly (code * scale; the
 * block's own K/V stay bf16).  Only the tcgen05 attention reads E4M3 caches:
 * a shape or model it does not take (more than 128 query rows per KV head,
 * head_dim other than 64/128, the mma.sync kernel selected at model
 * creation) gives DFLASH_ERR_UNSUPPORTED before any launch. */
int dflash_draft_block(dflash_model m, const int32_t* anchor, const int32_t* anchor_pos,
                       int32_t batch, const dflash_kv* kv, const void* pending_ctx,
                       const int32_t* pending_req, const int32_t* pending_pos, int32_t T,
                       int32_t* draft, float* logits, float* hidden, void* ws,
                       size_t ws_bytes, void* stream);

/* Shared LM head + argmax alone: argmax[r] = argmax_v (x[r] . lm_head[v]) for
 * `rows` rows of already final-normed hidden states x (bf16 [rows][hidden]);
 * lowest index on ties; optional fp32 logits [rows][vocab].  The same
 * kernels dflash_draft_block runs for its last step. */
int dflash_lm_head_argmax(dflash_model m, const void* x, int32_t rows, int32_t* argmax,
                          float* logits, void* ws, size_t ws_bytes, void* stream);

/* Greedy verify of `batch` requests, block size B (1..32).
 * draft int32 [batch][B-1]; target int32 [batch][B] (target[r][j-1] = the
 * target's argmax for block position j, i.e. t_j).
 * n = longest prefix with draft == target (0..B-1).  Outputs:
 *   out_tokens [batch][B]: t_1..t_{n+1}, then -1;   n_accept [batch];
 *   tgt_len_out = tgt_len_in + n + 1;  ctx_pending = n + 1;
 *   anchor_out = t_{n+1};  anchor_pos_out = anchor_pos_in + n + 1;
 *   ctx_pos [batch][B]: the positions of the block rows that become draft
 *   context (anchor and accepted drafts), anchor_pos_in + j for j <= n, then
 *   -1: the pending rows' positions for the next dflash_draft_block.
 * Any output may be NULL (not written); tgt_len_out, anchor_pos_out and
 * ctx_pos need their inputs.  In/out pairs may alias (ctx_pos must not alias
 * anchor_pos_in).  Pure integer work, bit-exact. */
int dflash_verify_greedy(const int32_t* draft, const int32_t* target, int32_t batch, int32_t B,
                         int32_t* out_tokens, int32_t* n_accept, const int32_t* tgt_len_in,
                         int32_t* tgt_len_out, int32_t* ctx_pending, int32_t* anchor_out,
                         const int32_t* anchor_pos_in, int32_t* anchor_pos_out, int32_t* ctx_pos,
                         void* stream);

/* Converts a bf16 cache (src, dtype 0) into an E4M3 cache (dst, dtype 1,
 * with scales) of the same geometry, for the model m: every position of every
 * page and layer (the layout and rounding are those of dflash_kv).  Pages and
 * page table are taken as they are; nothing but dst's pool and scales is
 * written.  DFLASH_ERR_INVALID_ARG (nothing launched): a null pointer, a pool
 * or scale array not 16-byte aligned, src not bf16, dst not E4M3, or page
 * counts that differ; DFLASH_ERR_UNSUPPORTED for a two-term cache.  src and
 * dst must not overlap. */
int dflash_kv_quantize(dflash_model m, const dflash_kv* src, const dflash_kv* dst, void* stream);

/* Verification at temperature T > 0 ("DFlash: how block diffusion boosts
 * NVIDIA Blackwell throughput", section "Real-world integration": sampling-
 * mode speedups; introduction: lossless).  The pages state no rule; this is
 * the standard lossless speculative-sampling rule applied per block
 * position, the drafts d_i having been drawn independently from
 * q_i = softmax(z_i / T) (dflash_sample_rows):
 *   accept d_i while u_i * q_i(d_i) < p_i(d_i), p_j = softmax(y_j / T);
 *   at the first rejection emit a draw from max(0, p_i - q_i), after B-1
 *   acceptances a draw from p_B.
 * draft int32 [batch][B-1]; draft_logits fp32 [batch][B][vocab] as
 * dflash_draft_block writes them (block row 0, the anchor, is not read; row
 * i+1 gives q for draft i); target_logits fp32 [batch][B][vocab] (row j-1 =
 * the target's logits for block position j); u fp64 [batch][B-1] acceptance
 * uniforms, w fp64 [batch][B] uniforms of the emitted draw at each position
 * (w[r][B-1]: the bonus); all in [0, 1).  A draw with uniform a returns the
 * smallest k with a*S < C_k (C the running sum of the weights, S the total).
 * Outputs as in dflash_verify_greedy; out_tokens is required, the others
 * may be NULL.  Arithmetic: fp32 exponentials of (z - max)/T, fp64 sums and
 * running sums in a fixed order, fp64 exp for the accept test; a decision
 * can differ from exact arithmetic only when its uniform lies within about
 * 1e-6 (relative) of the boundary.  Deterministic.  ws: 256-byte aligned,
 * at least dflash_sampling_workspace_bytes(batch, B), initialised with
 * dflash_workspace_init; a draft token outside [0, vocab) is rejected and
 * recorded as DFLASH_ERR_INVALID_ARG (site 401) in its status word.
 * batch >= 1, 1 <= B <= 32, temperature finite and > 0. */
size_t dflash_sampling_workspace_bytes(int32_t batch, int32_t B);
int dflash_verify_sampling(const int32_t* draft, const float* draft_logits,
                           const float* target_logits, int32_t batch, int32_t B, int32_t vocab,
                           double temperature, const double* u, const double* w,
                           int32_t* out_tokens, int32_t* n_accept, const int32_t* tgt_len_in,
                           int32_t* tgt_len_out, int32_t* ctx_pending, int32_t* anchor_out,
                           const int32_t* anchor_pos_in, int32_t* anchor_pos_out, int32_t* ctx_pos,
                           void* ws, size_t ws_bytes, void* stream);

/* Draft sampling for the temperature-T verify: one categorical draw from
 * softmax(z / T) per used row of logits fp32 [n_blocks][block][vocab] (with
 * skip_first = 1 the first row of every block is not used, as for the
 * drafter's anchor row); out int32 and a fp64 uniforms in [0, 1), both
 * indexed by used row ([n_blocks][block - skip_first]).  Same draw and
 * arithmetic as dflash_verify_sampling; ws as there, sized for
 * n_blocks*(block - skip_first) rows (64 KiB + 16 bytes per row). */
int dflash_sample_rows(const float* logits, int32_t n_blocks, int32_t block, int32_t skip_first,
                       int32_t vocab, double temperature, const double* a, int32_t* out,
                       void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------- end-to-end loop helpers */

/* Causal target forward over `batch` requests x `n` consecutive rows
 * (batch <= kv->n_rows, else DFLASH_ERR_CAPACITY before any launch):
 * tokens int32 [batch][n], row i of request r at position pos0[r] + i.  Each
 * row's K/V are written to the target cache at its position, then each row
 * attends to positions [0, pos0[r] + i] of its request.  tap_layers is a
 * HOST int32 array of n_taps distinct 0-indexed layers.  Outputs: argmax
 * int32 [batch][n]; optional taps bf16 [batch*n][n_taps*hidden] (residual
 * output of each listed layer, in list order); optional logits fp32
 * [batch*n][vocab].  A row's results do not depend on the other rows of the
 * call (fixed split-K and key-split boundaries), so a block verify and a
 * one-token-at-a-time decode give bit-identical tokens. */
int dflash_target_forward(dflash_model m, const int32_t* tokens, const int32_t* pos0,
                          int32_t batch, int32_t n, const dflash_kv* kv,
                          const int32_t* tap_layers, int32_t n_taps, void* taps,
                          int32_t* argmax, float* logits, void* ws, size_t ws_bytes,
                          void* stream);

/* Stand-in for the target's verify pass in draft-only benchmarks.  For block
 * position i = 1..B-1 of request r, target[r][i-1] = draft[r][i-1] when the top
 * 53 bits of h0 are below threshold[r] (agreement probability p_r as
 * floor(p_r * 2^53)), else (draft + 1 + h1 % (vocab-1)) % vocab; target[r][B-1]
 * = h1 % vocab; h0, h1 = splitmix64 output function of a key built from
 * (seed, *step, r, i, stream 0/1).  *step (device int64) is read, then
 * incremented by one when `advance` is non-zero. */
int dflash_synth_target(const int32_t* draft, int32_t batch, int32_t B,
                        const uint64_t* threshold, int32_t vocab, uint64_t seed,
                        int64_t* step, int32_t advance, int32_t* target, void* stream);

/* ------------------------------------------------------------ self-test */

/* Exercises the device-side failure path without faulting anything (not a
 * step of the method): one CTA waits, bounded by limit_ns, on an mbarrier in
 * its own shared memory that gets its single arrival only when `arrive` is
 * non-zero.  A wait that runs out records DFLASH_ERR_TIMEOUT with site 901 in
 * the workspace status word and the kernel returns normally, which is what
 * every bounded wait of the other kernels does (their limit is 1 s).
 * limit_ns: 1 .. 10^9.  waited_ns: device int64 (may be NULL), receives the
 * nanoseconds the wait took.  ws: an initialised workspace (only its status
 * word is used).  Bad arguments return DFLASH_ERR_INVALID_ARG before any
 * launch. */
int dflash_selftest_wait(int32_t arrive, int64_t limit_ns, int64_t* waited_ns, void* ws,
                         size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
