/*
 * dflash.h - C ABI of the DFlash drafter block step on one GB300 (sm_103a).
 *
 * The drafter is the block-diffusion draft model of DFlash speculative decoding
 * as the dflash-ops model card describes it (sections "Usage" and "Method") and
 * as dflash_head.rs lays out its weights (struct DflashLayer, struct
 * BlockDiffusionDraftHead): a few Qwen3-style layers that denoise a 16-token
 * block [anchor, mask x 15] in one non-causal forward, attending a per-layer
 * sliding-window ring of K/V injected from fused target-model features.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers; "host" pointers are
 *     ordinary process memory.  All device memory is owned by the caller and
 *     only borrowed by the library: weights, the ring, the scratch area and
 *     every input and output buffer must stay alive while a handle or a
 *     captured graph that names them can run.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *     stream.  Every call except dflash_create, dflash_read_status and
 *     dflash_step_host is asynchronous on that stream.
 *   - Matrices are row-major.  A weight W[out][in] computes y = x W^T.
 *   - Return value: DFLASH_OK (0) or a negative dflash_status.  Host-side
 *     checks run before anything is enqueued, so an error return means no
 *     work was launched.  DFLASH_ERR_CUDA keeps the CUDA error text in the
 *     handle (dflash_last_error).  No C++ exception crosses this boundary.
 *   - dflash_step and dflash_accept never allocate memory, never synchronise
 *     and never read device data on the host, so they can be captured in a
 *     CUDA graph (dflash_capture does exactly that).
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the library are exported explicitly (it is built with hidden
 * default visibility). */
#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

/* Rows of one noise block: the anchor token then 15 mask tokens
 * (dflash-ops model card, Method; the block size of the shipped drafter). */
#define DFLASH_BLOCK 16
/* Largest number of drafter layers a handle accepts (the shipped drafter has 5). */
#define DFLASH_MAX_LAYERS 16

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad enum value */
  DFLASH_ERR_UNSUPPORTED = -2,   /* geometry or dtype mix the library does not run */
  DFLASH_ERR_TOO_MANY_ROWS = -3, /* T > window, or T > max_inject */
  DFLASH_ERR_SEQ_RANGE = -4,     /* sequence index or n_seq outside [0, max_seq) */
  DFLASH_ERR_CUDA = -5,          /* a CUDA runtime call failed; see dflash_last_error */
  DFLASH_ERR_NOT_CAPTURED = -6,  /* dflash_replay before dflash_capture */
  DFLASH_ERR_DEVICE = -7         /* device status word non-zero (dflash_read_status) */
} dflash_status;

typedef enum {
  DFLASH_DTYPE_F32 = 0,
  DFLASH_DTYPE_BF16 = 1,
  DFLASH_DTYPE_FP8_E4M3 = 2,     /* E4M3 "fn" codes + one f32 scale per output row */
  /* E2M1 codes with one E4M3 scale per 16 weights of a row and one f32 scale per
   * row: w[n][k] = s[n] * e4m3(b[n][k/16]) * e2m1(q[n][k]).  A matrix [N][K] is
   * one buffer of N*K/2 code bytes (row-major) followed by N*K/16 block-scale
   * bytes; the row scales use the *_scale pointer.  Within each 16-byte group of
   * a row (32 weights) byte 4t + j holds the codes of k = 2(t + 4j) (low nibble)
   * and k + 1 (high nibble), t, j = 0..3.  Projection weights only
   * (q/k/v/o/gate/up/down, lm_head); every K (n_embd, n_head*head_dim, n_ff) a
   * multiple of 256.  The products run in fp16 against an fp16 hi/lo activation
   * pair (exact weights, activations to 2^-22 relative), so projection inputs
   * must stay below 65504 in magnitude.  dflash_head.rs (field lm_head_nvfp4)
   * names an NVFP4 LM head but not its layout: this one is the library's own. */
  DFLASH_DTYPE_FP4_E2M1 = 3
} dflash_dtype;

/* Bits of the device status word (dflash_read_status). */
#define DFLASH_DEV_BAD_TOKEN 0x1u     /* an id_last outside [0, n_vocab): clamped */
#define DFLASH_DEV_BAD_POSITION 0x2u  /* a negative inject position or n_past: row skipped */
#define DFLASH_DEV_TIMEOUT 0x4u       /* a pipeline wait gave up after ~2 s: outputs invalid */

/*
 * Drafter geometry and storage formats.
 *   n_layer <= DFLASH_MAX_LAYERS; n_head % n_head_kv == 0;
 *   head_dim in {32, 64, 128} (a multiple of 32 as the model card requires, and
 *   a divisor of the 128-row output tile of the projection kernels);
 *   n_embd, n_head*head_dim, n_ff and n_target_layers*target_embd multiples of 32.
 *   weight_dtype: q/k/v/o/gate/up/down and lm_head (F32, BF16 or FP8_E4M3);
 *   dense_dtype: tok_embd, fc, every norm weight and the target features
 *   (F32 or BF16); ring_dtype: ring K/V (F32 or BF16).
 *   max_seq: sequences (rings) the handle serves; max_inject: the largest row
 *   count of one dflash_encode / dflash_inject call (inject also needs
 *   T <= window: slots are pos % window, dflash-ops model card, Requirements).
 *   mask_token_id: token of block rows 1..15 (dflash_head.rs field mask_token_id).
 *   eps: RMSNorm epsilon (1e-6 in dflash_head.rs); rope_theta: rope base.
 */
typedef struct {
  int32_t n_layer;
  int32_t n_embd;
  int32_t n_head;
  int32_t n_head_kv;
  int32_t head_dim;
  int32_t n_ff;
  int32_t window;
  int32_t n_vocab;
  int32_t n_target_layers;
  int32_t target_embd;
  int32_t max_seq;
  int32_t max_inject;
  int32_t mask_token_id;
  int32_t weight_dtype;
  int32_t dense_dtype;
  int32_t ring_dtype;
  float eps;
  int32_t reserved0;
  double rope_theta;
} dflash_config;

/* One layer's device weights (dflash_head.rs, struct DflashLayer):
 *   attn_norm [n_embd], q_norm [head_dim], k_norm [head_dim], ffn_norm [n_embd]
 *     in dense_dtype;
 *   wq [n_head*head_dim][n_embd], wk and wv [n_head_kv*head_dim][n_embd],
 *   wo [n_embd][n_head*head_dim], gate and up [n_ff][n_embd], down [n_embd][n_ff]
 *     in weight_dtype;
 *   *_scale: f32 per output row, read only when weight_dtype is FP8_E4M3. */
typedef struct {
  const void* attn_norm;
  const void* wq;
  const void* wk;
  const void* wv;
  const void* wo;
  const void* q_norm;
  const void* k_norm;
  const void* ffn_norm;
  const void* gate;
  const void* up;
  const void* down;
  const float* wq_scale;
  const float* wk_scale;
  const float* wv_scale;
  const float* wo_scale;
  const float* gate_scale;
  const float* up_scale;
  const float* down_scale;
} dflash_layer_weights;

/* Model-level device weights:
 *   tok_embd [n_vocab][n_embd] dense_dtype and lm_head [n_vocab][n_embd]
 *     weight_dtype, both borrowed from the target model (dflash-ops model card,
 *     Usage); lm_head_scale f32 [n_vocab] for FP8;
 *   fc [n_embd][n_target_layers*target_embd], hidden_norm [n_embd],
 *   out_norm [n_embd] in dense_dtype (dflash_head.rs fields fc, hidden_norm, norm). */
typedef struct {
  const void* tok_embd;
  const void* lm_head;
  const float* lm_head_scale;
  const void* fc;
  const void* hidden_norm;
  const void* out_norm;
  dflash_layer_weights layers[DFLASH_MAX_LAYERS];
} dflash_weights;

typedef struct dflash_handle dflash_handle;

/*
 * Sizes of the two caller-owned device areas a handle needs.
 *   ring_bytes: K and V rings, [max_seq][n_layer][2][n_head_kv][window][head_dim]
 *     in ring_dtype, followed by ring_pos int32 [max_seq][window] (the position
 *     each slot holds, -1 when empty; one array per sequence, shared by layers).
 *   scratch_bytes: every intermediate of inject and step (activations, split-K
 *     partial sums, rope tables, counters, the status word).
 * Both areas must be 256-byte aligned.  Returns INVALID_ARG / UNSUPPORTED for a
 * bad configuration.
 */
DFLASH_API int dflash_workspace_size(const dflash_config* cfg, size_t* ring_bytes, size_t* scratch_bytes);

/*
 * Build a handle: validate the configuration, compute the host fp64 rope
 * inverse-frequency table theta^(-2j/head_dim) (dflash-ops model card, Method),
 * copy it into scratch, clear counters and the status word, zero the ring K/V
 * and mark every ring slot empty (ring_pos = -1).  Synchronous.  `w` is copied (the pointer
 * values, not the weights).  ring_mem and scratch_mem are device areas of at
 * least the dflash_workspace_size sizes.  On success *out receives the handle.
 */
DFLASH_API int dflash_create(const dflash_config* cfg, const dflash_weights* w, void* ring_mem,
                  void* scratch_mem, dflash_handle** out);

/* Free the handle's host state and its captured graph (not the borrowed memory). */
DFLASH_API void dflash_destroy(dflash_handle* h);

/*
 * Encode target features (dflash-ops model card, Usage: m.encode(target_features);
 * dflash_engine.py, class TargetContextFeatureFuser):
 *   H_t = RMSNorm(feats fc^T) * hidden_norm.
 *   feats: device [T][n_target_layers*target_embd] in dense_dtype;
 *   H_t:   device f32 [T][n_embd] (caller buffer, written).
 *   0 <= T <= max_inject (TOO_MANY_ROWS otherwise); T = 0 is a no-op.
 */
DFLASH_API int dflash_encode(dflash_handle* h, const void* feats, int32_t T, float* H_t, void* stream);

/*
 * dflash_encode for callers that cannot allocate device memory.  No page
 * defines this call; it exists for code that may not call cudaMalloc (an
 * allocator-free runtime, a plug-in limited to the buffers it is handed, a host
 * whose device memory is all owned by a pool) and therefore cannot provide the
 * scratch area dflash_create needs.  It computes exactly what dflash_encode
 * computes with the same kernels, without a handle:
 *   cfg:        geometry (n_embd, n_target_layers, target_embd, dense_dtype, eps;
 *               other fields are not read);
 *   fc:         device [n_embd][n_target_layers*target_embd], dense_dtype;
 *   hidden_norm: device [n_embd], dense_dtype;
 *   feats:      device [T][n_target_layers*target_embd], dense_dtype;
 *   H_t:        device f32 [T][n_embd], written (it also holds the intermediate
 *               un-normalised projection during the call).
 * Its intermediate memory is one 8 MiB file-scope __device__ array that every
 * GPU loading this library holds until the process exits.  Limits: with
 * tiles = ceil(n_embd / 128), tiles * ceil(T / 16) <= 16384 and
 * tiles * T <= 835,584 (T <= 5040 at n_embd 6656); larger calls return
 * DFLASH_ERR_TOO_MANY_ROWS and launch nothing.  The first call on a device looks
 * up the array's device address and sets kernel attributes for that device
 * (the device current at the call); make that first call before any stream
 * capture.  Nothing is allocated or freed, by this library or any library it
 * calls.  All calls share the array: calls that overlap on the GPU (on
 * different streams, or from different threads) race; it is cleared where it
 * must start at zero at the start of every call.  Asynchronous on `stream`.
 * There is no handle to hold an error text: DFLASH_ERR_CUDA from this call
 * carries no further detail (the runtime's own cudaGetLastError does).  The
 * runtime's last-error slot is cleared on entry, so an error left by earlier
 * unrelated work is not reported as this call's.
 */
DFLASH_API int dflash_encode_noalloc(const dflash_config* cfg, const void* fc, const void* hidden_norm,
                                     const void* feats, int32_t T, float* H_t, void* stream);

/*
 * Inject encoded rows into sequence `seq`'s ring (dflash-ops model card, Method
 * and Requirements): for every layer l and row t,
 *   K = rope(RMSNorm_head(H_t[t] wk_l^T) * k_norm_l, pos[t]),  V = H_t[t] wv_l^T,
 *   both rounded once to ring_dtype and stored at slot pos[t] % window, and
 *   ring_pos[slot] = pos[t].  No attn_norm is applied to H_t.
 *   H_t: device f32 [T][n_embd]; pos: device int32 [T], non-negative and
 *   distinct modulo window (contiguous positions are).  0 <= T <= min(window,
 *   max_inject); seq in [0, max_seq).  A negative position sets
 *   DFLASH_DEV_BAD_POSITION and its row is skipped.
 */
DFLASH_API int dflash_inject(dflash_handle* h, int32_t seq, const float* H_t, const int32_t* pos,
                  int32_t T, void* stream);

/*
 * Block width of the following steps, accepts, loop turns and captures
 * (dflash_head.rs, set_block_g: the scheduler's narrower block of the anchor
 * plus num_drafts mask rows, clamped to 2..16; its propose graphs are keyed by
 * width because a capture bakes its row count).  With width B the block holds
 * rows 0..B-1 at positions n_past .. n_past+B-1 ([id_last, mask x (B-1)]),
 * every row attends to the B block keys (and the ring); drafts j >= B-1 are
 * written as -1; logits rows >= B are computed but are not part of the result;
 * accept and advance count at most B-1 drafts.  dflash_capture and
 * dflash_capture_loop store one graph per width, and dflash_replay launches
 * the current width's graph.  2 <= width <= 16 (INVALID_ARG otherwise, or
 * while a capture is running).  Default 16.
 */
DFLASH_API int dflash_set_block_width(dflash_handle* h, int32_t width);

/*
 * Projection chains (off by default).  With chains on, a step of fewer than
 * 128 block rows with bf16, fp32 or E4M3 weights runs, per layer, one
 * persistent launch for o, gate/up, down and the next layer's q/k/v (the LM
 * head after the last layer) instead of four (dflash-ops model card,
 * Requirements and limits: the whole-block megakernel is the named next step;
 * this is its projection part).  Its CTAs wait for one another's output tiles
 * (bounded waits that end in DFLASH_DEV_TIMEOUT), which needs the whole grid
 * resident at once: keep chains off when other work may hold SMs for the
 * duration of a step (a GPU shared through MPS or partitioned contexts).
 * Results are bitwise identical either way; on a GB300 the chained step is not
 * faster (every tile of a stream-K phase completes near the phase's end, so the
 * next phase starts no earlier than after a kernel boundary with programmatic
 * dependent launch).  enable = 0 or 1; UNSUPPORTED when enabling on a handle
 * without chains (FP4 or E4M3 weights, or a device that cannot hold the grid);
 * INVALID_ARG during a capture.  Takes effect for later steps and captures.
 */
DFLASH_API int dflash_set_chain(dflash_handle* h, int32_t enable);

/*
 * The attention kernel a step of n_seq sequences runs (the choice is
 * automatic; this reports it for tests and benchmarks): 0 = split window (the
 * window of every (sequence, kv head) in 128-slot CTAs that the GPU holds at
 * once, merged through global scratch), 1 = clusters (a kv head's window over
 * up to 8 CTAs of a cluster, merged through distributed shared memory), 2 =
 * stream-K (one CTA per SM streaming equal ranges of all windows through a
 * double-buffered TMA pipeline; windows cut by a range merge their partials).
 * Returns the kind, INVALID_ARG for a null handle, SEQ_RANGE for n_seq outside
 * 1..max_seq.
 */
DFLASH_API int dflash_attention_kernel(const dflash_handle* h, int32_t n_seq);

/*
 * One block step for sequences 0..n_seq-1 (dflash-ops model card, Usage:
 * step(id_last, n_past) -> logits [16, n_vocab]; drafts = argmax of rows 1..15).
 *   id_last: device int32 [n_seq], the anchor token of each block;
 *   n_past:  device int32 [n_seq], position of block row 0 (rows sit at
 *            n_past .. n_past+15; ring slots holding positions p with
 *            0 <= p < n_past and n_past + i - p < window are row i's keys;
 *            all 16 block rows are keys of every row);
 *   logits:  device f32 [n_seq][16][n_vocab] (written), or NULL to skip storing
 *            them (drafts are still computed);
 *   drafts:  device int32 [n_seq][15], argmax of block rows 1..15, ties to the
 *            lowest token id (written).
 * 1 <= n_seq <= max_seq.  Scalars are read on the device, so a captured graph
 * replays with new id_last / n_past contents.
 */
DFLASH_API int dflash_step(dflash_handle* h, int32_t n_seq, const int32_t* id_last, const int32_t* n_past,
                float* logits, int32_t* drafts, void* stream);

/*
 * First-mismatch acceptance scan on the device (dflash-ops model card, Usage:
 * n_ok = m.accept(drafts, target_tokens); dflash_engine.py,
 * DFlashSpeculativeVerifier.verify_block): n_ok[s] = the number of leading
 * j in 0..14 with drafts[s][j] == targets[s][j] (15 when all agree).
 *   drafts, targets: device int32 [n_seq][15]; n_ok: device int32 [n_seq].
 */
DFLASH_API int dflash_accept(dflash_handle* h, int32_t n_seq, const int32_t* drafts, const int32_t* targets,
                  int32_t* n_ok, void* stream);

/*
 * Capture dflash_step (and dflash_accept when targets and n_ok are non-NULL)
 * with these exact pointers into a CUDA graph owned by the handle (dflash-ops
 * model card, Method: the captured step allocates nothing, so eager work may
 * run between replays).  Capture runs on an internal stream; nothing is
 * launched.  `stream` orders the capture after earlier work on it.
 * Replaces a previous dflash_capture of the current block width (a loop-turn
 * graph of dflash_capture_loop is kept separately and is not affected).
 */
DFLASH_API int dflash_capture(dflash_handle* h, int32_t n_seq, const int32_t* id_last, const int32_t* n_past,
                   float* logits, int32_t* drafts, const int32_t* targets, int32_t* n_ok,
                   void* stream);

/* Launch the current width's dflash_capture graph on `stream` (NOT_CAPTURED if there is none). */
DFLASH_API int dflash_replay(dflash_handle* h, void* stream);

/*
 * Node counts of the current width's captured graph (loop = 0: dflash_capture,
 * loop != 0: dflash_capture_loop), host int32 outputs: kernel launches, memory
 * allocation or free nodes (always 0: nothing in a step allocates), and every
 * other node (memset nodes of profiling captures).  NOT_CAPTURED if there is no
 * such graph.
 */
DFLASH_API int dflash_graph_nodes(dflash_handle* h, int32_t loop, int32_t* kernels,
                                  int32_t* mem_alloc, int32_t* other);

/*
 * One turn of the speculative loop on the device, after the target model has
 * verified the block that the last dflash_step drafted (dflash_engine.py,
 * DFlashSpeculativeVerifier.verify_block: accepted prefix + one bonus token;
 * dflash-ops model card, Usage: inject(encode(features), positions) of the
 * verified positions, then the next step(id_last, n_past)).  Per sequence s:
 *   m = number of leading j in 0..14 with drafts[s][j] == targets[s][j];
 *   the target features of block rows 0..m (positions n_past[s] .. n_past[s]+m)
 *   are encoded and injected into sequence s's ring (rows m+1..15 are encoded
 *   but not written: their slots may still hold keys inside the window);
 *   n_ok[s] = m; id_last[s] = targets[s][m] (the target's own token after the
 *   accepted drafts: the correction, or the bonus token when m = 15);
 *   n_past[s] += m + 1.
 *   drafts:  device int32 [n_seq][15] (the previous step's drafts);
 *   targets: device int32 [n_seq][16], the target's greedy token at block rows
 *            0..15 (row j predicts position n_past + j + 1);
 *   feats:   device [n_seq][16][n_target_layers*target_embd] in dense_dtype,
 *            the target's features at block rows 0..15;
 *   id_last, n_past: device int32 [n_seq], read and updated in place;
 *   n_ok:    device int32 [n_seq], written.
 * Requires 16 * n_seq <= max_inject and window >= 16 (TOO_MANY_ROWS
 * otherwise).  Nothing is read back to the host, so the call can be captured
 * (dflash_capture_loop).  Asynchronous on `stream`.
 */
DFLASH_API int dflash_advance(dflash_handle* h, int32_t n_seq, const int32_t* drafts,
                              const int32_t* targets, const void* feats, int32_t* id_last,
                              int32_t* n_past, int32_t* n_ok, void* stream);

/*
 * Capture one whole loop turn - dflash_advance followed by dflash_step with
 * the updated id_last / n_past - into the handle's loop graph of the current
 * block width (replacing a previous loop capture of that width; a dflash_capture
 * graph is kept separately; dflash_replay_loop launches it).  With these exact pointers,
 * each replay consumes the target's tokens and features for the block drafted
 * by the previous replay (or step) and leaves the next block's logits and
 * drafts in `logits` / `drafts`.  Capture runs on an internal stream; nothing
 * is launched; `stream` orders the capture after earlier work on it.
 */
DFLASH_API int dflash_capture_loop(dflash_handle* h, int32_t n_seq, const int32_t* targets,
                                   const void* feats, int32_t* id_last, int32_t* n_past,
                                   int32_t* n_ok, float* logits, int32_t* drafts, void* stream);

/* Launch the current width's dflash_capture_loop graph on `stream` (NOT_CAPTURED if there is none). */
DFLASH_API int dflash_replay_loop(dflash_handle* h, void* stream);

/*
 * The same step as dflash_step, driven from host memory: copies id_last and
 * n_past (host int32 [n_seq]) to the device, runs the step into internal
 * scratch buffers, copies the drafts back to host int32 [n_seq][15] (and the
 * logits to host f32 [n_seq][16][n_vocab] when `logits` is non-NULL), and waits
 * for `stream`.  Host buffers may be pageable or pinned.
 */
DFLASH_API int dflash_step_host(dflash_handle* h, int32_t n_seq, const int32_t* id_last,
                     const int32_t* n_past, float* logits, int32_t* drafts, void* stream);

/* Zero sequence `seq`'s ring K/V and mark every slot empty (ring_pos = -1), on `stream`. */
DFLASH_API int dflash_ring_reset(dflash_handle* h, int32_t seq, void* stream);

/*
 * Read and clear the device status word (DFLASH_DEV_* bits) after waiting for
 * `stream`.  Synchronous.  Returns DFLASH_ERR_DEVICE when a bit was set.
 */
DFLASH_API int dflash_read_status(dflash_handle* h, uint32_t* status, void* stream);

/*
 * Profiling.  dflash_profile_enable(h, mode): 0 off; 1 launch-class events on
 * eager calls; 2 device timestamps of every step launch.
 *
 * Mode 1 (eager calls, not captured graphs): every kernel launch of
 * dflash_step / dflash_encode / dflash_inject / dflash_accept is bracketed by
 * CUDA events recorded on the launching stream.
 * dflash_profile_read waits for those events, writes the summed device time in
 * milliseconds and the launch count of each class (arrays of DFLASH_PROF_N
 * entries, host memory) and clears the record.  Classes: 0 embedding + rope
 * table, 1 q/k/v projection, 2 attention chunks, 3 attention merge, 4 o
 * projection, 5 gate/up projection, 6 down projection, 7 LM head + drafts,
 * 8 encode (fc + norm), 9 injection (rope table + wk/wv + ring scatter),
 * 10 acceptance scan, 11 projection chain (one launch of o, gate/up, down and
 * the next layer's q/k/v or the LM head: steps of fewer than 128 block rows
 * with bf16, fp32 or E4M3 weights).  Enabling while a capture is in progress
 * is refused.
 */
#define DFLASH_PROF_N 12
DFLASH_API int dflash_profile_enable(dflash_handle* h, int enable);
DFLASH_API int dflash_profile_read(dflash_handle* h, double* ms, int32_t* launches);

/*
 * Mode 2: every kernel of a step (and of the acceptance scan of dflash_capture)
 * records the %globaltimer of its first CTA's start and of its last CTA's end
 * in a scratch slot, from eager calls and from graphs captured while mode 2 is
 * on (such a graph also zeroes the slots with one memset node ahead of the
 * step); the kernels, their order and their launch attributes are those of the
 * unprofiled step.  dflash_profile_stamps waits for `stream`, then writes, for
 * the launches of the last recorded step in launch order (at most `max`), the
 * class (as in mode 1) and the start and end in microseconds relative to the
 * earliest start (-1 for a launch that has not run), and their count to *n
 * (host arrays).  Synchronous.
 */
DFLASH_API int dflash_profile_stamps(dflash_handle* h, int32_t max, int32_t* cls, double* start_us,
                                     double* end_us, int32_t* n, void* stream);

/* Text of a dflash_status code (static storage). */
DFLASH_API const char* dflash_status_string(int status);

/* Text of the last CUDA error recorded in the handle ("" if none). */
DFLASH_API const char* dflash_last_error(const dflash_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
