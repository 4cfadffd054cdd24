/*
 * ff.h -- C ABI of libff.so: the renderer bank-attention hot path of
 * FlashForward on one GB300 (sm_103a).
 *
 * Source of the operation: "FlashForward가 디노이징 중 KV 캐시를 재사용해 자기회귀
 * 영상 생성을 가속한다" (onedev.kr/papers/332), section "어떻게 동작하나" (how it
 * works), Eq. (2):
 *     (v_hat, K, V) = F_R(x, c, tau_k; A_Gamma(i), B_k^(i))
 *     B_k^(i+1)    = Tail_H(B_k^(i) U (i, K, V))
 * The renderer forward of chunk i at denoising stage k reads the clean-anchor
 * KV chosen by Gamma(i) and the stage-matched KV of the last H chunks, and
 * publishes its own in-flight K/V into the same stage bank; there is no
 * cache-update-only forward.  Anchors: section "무엇과 다른가" (stride Delta,
 * planner blocks of 3, cache-extraction forward per block).
 *
 * This library implements the attention part of F_R for one transformer
 * layer per call: rotary position encoding of the chunk's Q/K, publish of
 * (K, V) into the stage bank, and softmax(Q K^T / sqrt(d)) V over the context
 * [anchors of Gamma(i); last H chunks of the stage; own chunk].  The context
 * is never copied into one buffer: the attention kernel's TMA tensor loads
 * read the anchor slots and the stage-ring slots where they live.
 *
 * Conventions for every entry point:
 *  - Tensors are bf16, row-major [tokens, heads, head_dim] with tokens
 *    frame-major and each latent frame row-major over (y, x).  Pointers are
 *    DEVICE pointers of the bank's device unless stated otherwise, 16-byte
 *    aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on it; inputs must stay valid and
 *    outputs must not be read until the stream has passed the call.
 *  - The caller owns all input/output buffers and streams; the bank owns all
 *    memory it allocates.  No call allocates device memory after
 *    ff_bank_create.
 *  - Every call returns an ff_status.  On any error the bank state is left
 *    unchanged.  Argument, order and residency errors are found before any
 *    work is enqueued.  FF_ERR_CUDA from a kernel launch that fails after an
 *    earlier kernel of the same call was enqueued (ff_render_attn: the
 *    publish kernel runs before the attention kernel) leaves that earlier
 *    work enqueued; it wrote only memory that no resident chunk occupies, so
 *    the observable bank state is still unchanged.  Nothing aborts the
 *    process.
 *  - A bank may be used from one host thread at a time.
 */
#ifndef FF_H_
#define FF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ff_status {
  FF_OK = 0,
  FF_ERR_ARG = 1,             /* null pointer, index out of range, unsupported shape */
  FF_ERR_ORDER = 2,           /* chunk != next chunk of (layer, stage): calls are sequential */
  FF_ERR_ANCHOR_MISSING = 3,  /* an anchor of Gamma(i) was never published or was evicted */
  FF_ERR_OOM = 4,             /* device allocation failed or would exceed desc.max_bytes */
  FF_ERR_CUDA = 5,            /* a CUDA runtime call failed */
  FF_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait gave up (reported by ff_bank_error_poll) */
  FF_ERR_UNSUPPORTED = 7      /* device is not compute capability 10.3 */
} ff_status;

/* Bank description (plain old data).  Defaults from ff_desc_default follow
 * the pages' experiment settings (onedev.kr/papers/332, "무엇과 다른가":
 * B_R = 3, Delta = 10, S = 4, H = 5). */
typedef struct ff_bank_desc {
  int n_layers;         /* transformer layers, each with its own banks (>= 1) */
  int n_stages;         /* S denoising stages = stage banks per layer (>= 1) */
  int history;          /* H: chunks kept per stage bank (>= 1) */
  int chunk_frames;     /* B_R: latent frames per renderer chunk (1..8) */
  int anchor_stride;    /* Delta: latent frames between clean anchors (>= 1) */
  int anchor_capacity;  /* slots of the per-layer anchor ring; anchor a -> slot (a/Delta) mod capacity */
  int total_frames;     /* N latent frames of the video */
  int heads;            /* attention heads h */
  int head_dim;         /* d: 64 or 128 */
  int frame_h;          /* latent frame height in tokens (rows, y) */
  int frame_w;          /* latent frame width in tokens (columns, x); tokens per frame T = frame_h * frame_w */
  double rope_theta;    /* rotary base theta (10000) */
  size_t max_bytes;     /* 0 = unlimited; otherwise create fails with FF_ERR_OOM above this many device bytes */
  int device;           /* CUDA device ordinal */
  int planner_block;    /* B_P: anchors per planner block (default 3) */
  int planner_history;  /* H_P: previous planner blocks a planner block attends to (default 6; 0 = no planner scratch) */
} ff_bank_desc;

typedef struct ff_bank ff_bank_t;

/* Fill `d` with the defaults above (n_layers 1, N 81, 12 heads, d 128,
 * 30 x 52 tokens, 9 anchor slots, device 0). */
int ff_desc_default(ff_bank_desc* d);

/* Allocate every device buffer the bank will ever use: the stage rings
 * (H + 1 physical chunk slots per (layer, stage), so that chunk i can be
 * written while chunks i-H .. i-1 are read in place) and the anchor ring of
 * every layer, per-stage rotated-Q scratch and attention split partials, the
 * planner scratch and the rotary tables.  Returns
 * FF_ERR_ARG for an invalid description, FF_ERR_UNSUPPORTED if the device
 * is not sm_103, FF_ERR_OOM if the total exceeds max_bytes or an allocation
 * fails (nothing stays allocated then).  *out is set only on FF_OK. */
int ff_bank_create(const ff_bank_desc* desc, ff_bank_t** out);

/* Publish the clean anchor KV of `n_anchors` consecutive anchors
 * first_anchor_frame, + Delta, ... (a planner block's cache-extraction
 * forward; onedev.kr/papers/332, "무엇과 다른가").  k_pre, v: device bf16
 * [n_anchors * T, heads, head_dim], anchor-major.  K is rotated at
 * t = anchor frame and stored with V in slot (a / Delta) mod capacity of
 * `layer`, replacing what that slot held.  Errors: FF_ERR_ARG if the first
 * frame is not a multiple of Delta, the last anchor is past the video, or
 * n_anchors is not in 1..anchor_capacity. */
int ff_anchor_publish(ff_bank_t* bank, int layer, int first_anchor_frame, int n_anchors,
                      const void* k_pre, const void* v, void* stream);

/* Renderer bank attention of chunk `chunk` at stage `stage` of `layer`
 * (Eq. (2) above).  q_pre, k_pre, v: device bf16 [F_i * T, heads, head_dim],
 * F_i = frames of the chunk (B_R, or fewer for the last chunk), before
 * rotary encoding.  out: device bf16 of the same shape,
 * out = softmax(RoPE(Q) K_ctx^T / sqrt(d)) V_ctx per head, where the context
 * is [Gamma(i) anchors; chunks max(0, i-H) .. i-1 of this stage; own chunk].
 * Afterwards slot i mod H of (layer, stage) holds (i, RoPE(K), V).
 * Errors: FF_ERR_ORDER unless chunk equals the next chunk of (layer, stage)
 * (0, 1, 2, ... in order); FF_ERR_ANCHOR_MISSING if an anchor of Gamma(i) is
 * not resident. */
int ff_render_attn(ff_bank_t* bank, int layer, int stage, int chunk,
                   const void* q_pre, const void* k_pre, const void* v, void* out, void* stream);

/* One renderer call of a batch: the arguments of ff_render_attn. */
typedef struct ff_render_call {
  int layer;
  int stage;
  int chunk;
  const void* q_pre;
  const void* k_pre;
  const void* v;
  void* out;
} ff_render_call;

/* n independent renderer calls issued together (1 <= n <= 4, one call per
 * stage: the stages of the calls are distinct).  The result, the bank state
 * afterwards and every error are those of calling ff_render_attn for
 * calls[0], ..., calls[n-1] in order; since each call reads and writes only
 * its own stage bank (and reads resident anchors), the calls do not depend on
 * each other.  This is the single-GPU form of the pages' stage wavefront
 * (onedev.kr/papers/332, "어떻게 동작하나": the S denoising stages work on
 * different in-flight chunks at once, stage k on chunk i - k): the S calls of
 * one layer at one wavefront step are independent.  All calls' RoPE/publish
 * items run as one launch and all their query blocks as one attention launch,
 * so the work of the calls is balanced across the SMs together.  Any error is
 * found before any work is enqueued (FF_ERR_ARG also for n out of range or a
 * repeated stage); the state is then unchanged. */
int ff_render_attn_batch(ff_bank_t* bank, int n, const ff_render_call* calls, void* stream);

/* Planner-role attention of planner block `block` of `layer`
 * (onedev.kr/papers/332, "무엇과 다른가": the planner produces the clean anchors
 * B_P = 3 at a time with history H_P = 6 and context budget W_ctx = 21;
 * "어떻게 쓰나": planner blocks attend causally to the clean KV of previous
 * blocks).  Block b holds anchors b*B_P .. b*B_P + B_P - 1 (frames a*Delta;
 * fewer in the last block).  q_pre, k_pre, v: device bf16
 * [n_b * T, heads, head_dim] for the block's n_b anchor frames, before rotary
 * encoding; out: same shape, out = softmax(RoPE(Q) K_ctx^T / sqrt(d)) V_ctx
 * with context [clean anchor KV of blocks max(0, b - H_P) .. b-1, oldest first;
 * the block itself], i.e. at most H_P * B_P + B_P = W_ctx frames.  Nothing is
 * published: the block's clean KV enters the anchor ring through
 * ff_anchor_publish once the block is done.  Errors: FF_ERR_ARG (block out of
 * range, planner_history == 0), FF_ERR_ANCHOR_MISSING if an anchor of the
 * history blocks is not resident (size anchor_capacity >= H_P * B_P). */
int ff_planner_attn(ff_bank_t* bank, int layer, int block, const void* q_pre, const void* k_pre, const void* v,
                    void* out, void* stream);

/* Packed block-causal renderer forward of one denoising stage: every chunk of
 * the video in one call (onedev.kr/papers/332, "어떻게 쓰나": in training the
 * renderer runs as a block-causal forward rather than chunk-by-chunk cache
 * updates; its targets attend to the Gamma(i) clean anchor KV and the previous
 * H same-noise-level chunks).  Rows of chunk i attend to [Gamma(i) anchors;
 * chunks max(0, i-H) .. i-1; chunk i], exactly the key set ff_render_attn uses
 * for chunk i when the chunks are rendered in order at one stage.
 * q_pre, k_pre, v: device bf16 [N * T, heads, head_dim] for all N latent frames,
 * before rotary encoding; anchor_k_pre, anchor_v: [A * T, heads, head_dim] for
 * the A anchors 0, Delta, 2 Delta, ...; out: [N * T, heads, head_dim].
 * workspace: device buffer of at least ff_packed_workspace_bytes bytes, owned by
 * the caller (rotated K, V of anchors and frames and rotated Q).  Uses the bank's
 * description and rotary tables only: no bank state is read or changed.
 * Errors: FF_ERR_ARG for null/misaligned pointers or a short workspace. */
int ff_packed_workspace_bytes(const ff_bank_t* bank, size_t* bytes);
int ff_packed_render_attn(ff_bank_t* bank, const void* q_pre, const void* k_pre, const void* v,
                          const void* anchor_k_pre, const void* anchor_v, void* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Wait for all work the bank enqueued, then free everything.  NULL-safe. */
int ff_bank_destroy(ff_bank_t* bank);

/* ---- introspection (used by tests; host-side, no device work unless stated) ---- */

/* Gamma(i): left anchor, right anchor (-1 if none) and their count. */
int ff_bank_gamma(const ff_bank_t* bank, int chunk, int* left, int* right, int* n);

/* Slot state.  stage >= 0: slot `slot` (0..H-1) of the stage bank; stage == -1:
 * slot of the anchor ring.  chunk_tag = chunk index (stage bank) or anchor
 * frame (anchor ring), -1 if empty; frames = latent frames held; k, v =
 * device pointers to the slot's bf16 [frames * T, heads, head_dim] data
 * (valid for the bank's lifetime; contents change with later calls). */
int ff_bank_slot_info(const ff_bank_t* bank, int layer, int stage, int slot, int* chunk_tag,
                      int* frames, const void** k, const void** v);

/* Device bytes owned by the bank (constant from create to destroy). */
int ff_bank_bytes(const ff_bank_t* bank, size_t* bytes);

/* Synchronise the bank's device and read the device error word: FF_OK or
 * FF_ERR_DEVICE_TIMEOUT (a bounded wait in a kernel gave up; that call's
 * output is undefined).  Clears the word. */
int ff_bank_error_poll(ff_bank_t* bank);

/* Static description of a status code. */
const char* ff_status_string(int status);

/* ---- host-only planning (no device needed) ---- */

typedef struct ff_chunk_plan {
  int first_frame;      /* first latent frame of the chunk */
  int n_frames;         /* frames of the chunk */
  int n_anchors;        /* 1 or 2 */
  int anchors[2];       /* Gamma(i), left first */
  int n_hist;           /* history chunks (min(i, H)) */
  int hist_first;       /* oldest history chunk */
  int hist_frames;      /* frames in the history chunks */
  int slot;             /* stage-bank slot the chunk publishes into (i mod H) */
  int key_frames;       /* anchors + history + own frames */
} ff_chunk_plan;

/* Chunk plan of `chunk` for a description (FF_ERR_ARG past the last chunk). */
int ff_plan_chunk(const ff_bank_desc* desc, int chunk, ff_chunk_plan* out);

typedef struct ff_planner_plan {
  int first_anchor;     /* first anchor index of the block (frame = index * Delta) */
  int n_anchors;        /* anchors in the block (B_P, fewer at the end) */
  int hist_first_block; /* oldest history block */
  int n_hist_blocks;    /* min(block, H_P) */
  int hist_frames;      /* anchor frames of the history blocks */
  int key_frames;       /* hist_frames + n_anchors */
} ff_planner_plan;

/* Plan of planner block `block` (FF_ERR_ARG past the last block). */
int ff_plan_planner_block(const ff_bank_desc* desc, int block, ff_planner_plan* out);

/* ---- timing of the library's own kernels (CUDA events on the call's stream) ---- */

typedef struct ff_kernel_times {
  int calls;            /* renderer calls timed since the last reset (a batch counts its calls) */
  double publish_ms;    /* summed duration of the RoPE + publish launches */
  double attn_ms;       /* summed duration of the attention launches */
  double combine_ms;    /* summed duration of the split-combine launches (0 when unsplit) */
  int launches;         /* kernels launched by the timed calls */
} ff_kernel_times;

/* enable != 0: record events around each kernel launch of subsequent renderer
 * calls (ff_render_attn, ff_render_attn_batch).  Resets the accumulated times.
 * Synchronises the bank's device; the events are created here (2048 calls'
 * worth, and that many more whenever a run of timed calls without a reset
 * needs them), so timed calls record into existing events.  Returns
 * FF_ERR_CUDA if the events cannot be created. */
int ff_bank_set_timing(ff_bank_t* bank, int enable);

/* Synchronise on the recorded events and return the accumulated times. */
int ff_bank_read_timing(ff_bank_t* bank, ff_kernel_times* out);

/* Number of kernels one ff_render_attn call of `chunk` launches (2 or 3). */
int ff_render_kernel_count(const ff_bank_t* bank, int chunk, int* count);

/* ---- self-test of failure detection ----
 *
 * Enqueue one small kernel whose bounded wait can never be satisfied: it
 * gives up after limit_ms (1..10000) and sets the bank's device error word,
 * exactly as a render kernel does when one of its waits runs out.  Used to
 * test that ff_bank_error_poll reports FF_ERR_DEVICE_TIMEOUT without
 * faulting or hanging the GPU; the context stays usable afterwards. */
int ff_bank_wait_probe(ff_bank_t* bank, int limit_ms, void* stream);

/* ---- attention without any device allocation ----
 *
 * The pages have no counterpart of this entry point.  It serves callers that
 * cannot call cudaMalloc: code running inside a CUDA stream capture, hosts
 * whose memory is owned by another allocator, processes that must not grow
 * their device footprint after start-up.  Such a caller holds the rotated
 * queries and the gathered context itself and needs only the attention step.
 *
 * out = softmax(q k^T / sqrt(head_dim)) v per head, computed by the same
 * tcgen05 kernel as ff_render_attn.  q, out: device bf16 [nq, heads, head_dim];
 * k, v: device bf16 [nk, heads, head_dim]; all 16-byte aligned, owned by the
 * caller, on the current device; head_dim 64 or 128.  Asynchronous on `stream`
 * (a cudaStream_t of the current device).
 *
 * Scratch: key-range split partials live in one static device array of
 * FF_NOALLOC_SCRATCH_BYTES, created when the library's module loads on a
 * device and kept until the process exits.  The work plan is the bank path's
 * (whole units first, the rest cut into up to 4 key ranges), restricted to
 * plans whose partials fit: a split plan needs
 * 256 + split_units * n_split * 256 * (4 * head_dim + 8) bytes, and the plan
 * without a split needs none, so no problem is refused for its size.  Sizes
 * beyond the kernels' index limits (more than 2^24 key tiles of 128 or
 * (head, 256-row query block) units, or 2^31 elements per tensor) are refused
 * with FF_ERR_ARG before any work is enqueued.  The first call on a device
 * (that device current) sets up the array's address and the kernel
 * attributes: make it before any stream capture.  All calls share the array,
 * so calls that overlap on the GPU race; order them on one stream.  A bounded
 * device wait that gives up leaves `out` undefined and is not reported by
 * this entry point.  Returns FF_OK, FF_ERR_ARG (also for a stream of another
 * device), FF_ERR_CUDA or FF_ERR_UNSUPPORTED (device not sm_103). */
#define FF_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int ff_attention_noalloc(const void* q, const void* k, const void* v, void* out, int nq, int nk, int heads,
                         int head_dim, void* stream);

#ifdef __cplusplus
}
#endif

#endif  /* FF_H_ */
