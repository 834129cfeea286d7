/*
 * kvring -- a rolling FP8 attention cache for one GPU (sm_103a).
 *
 * One kvring_t holds one transformer layer's attention cache, as described
 * in "Runway Characters: Serving a 57B Video Diffusion Transformer for
 * Real-Time Conversation" (Runway research post):
 *
 *   - section "Do It Once, at Write Time": each new frame's keys get rotary
 *     position embeddings (RoPE) once, as they enter the cache, and keys and
 *     values are quantised to FP8 with per-head scales calibrated once per
 *     session; the cache is a ring, so the window advances by overwriting
 *     the oldest slots with no copy; at each periodic position reset a
 *     single delta rotation is applied to the cached keys in place; after
 *     wrap-around slot order is not time order, so every slot keeps its own
 *     position;
 *   - section "Where the Time Went": every attention call reads its layer's
 *     cache (5,788 slots, 757 of them new);
 *   - sections "What Broke in Production" and "Blackwell and Beyond Four
 *     GPUs": no host/device synchronisation on the steady path, no buffer
 *     per input shape, calls that chain correctly inside CUDA graphs, and an
 *     FP8 attention kernel that takes per-head scales.
 *
 * Formats.  FP8 is OCP OFP8 E4M3 ("fn": bias 7, no infinities, largest
 * finite 448), rounded to nearest even with saturation to +-448.  RoPE is
 * the adjacent-pair form: pair (x[2i], x[2i+1]) rotates by p * base^(-2i/d).
 *
 * Conventions for every entry point.
 *   - Tensors are device pointers, row-major and contiguous, 16-byte
 *     aligned.  Token inputs are bf16 [n][num_heads][head_dim] (what a QKV
 *     projection emits).  Positions are int32 [n] on the device.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on that stream; none synchronises with the
 *     host, none allocates memory.  Calls on one ring must be ordered (one
 *     stream, or the caller's events); two rings are independent.
 *   - A ring belongs to the device that was current at kvring_create; every
 *     call that takes a ring returns KVRING_ERR_INVALID_ARG unless that
 *     device is current (the kernels would otherwise run on another GPU
 *     against this one's memory).  Its tensors and stream must be on that
 *     device too, which the library cannot check.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     failed check enqueues nothing and returns an error status.  CUDA
 *     launch failures return KVRING_ERR_CUDA.  Problems only the device can
 *     see (a position outside the RoPE table, a timed-out wait) set bits in
 *     an error word that kvring_export() returns in state[KVRING_STATE_ERROR];
 *     the kernels then skip the offending element instead of faulting.
 *   - The ring's head, fill level and next position live in device memory,
 *     so a CUDA graph that captured a write or an attention call advances
 *     the ring correctly on every replay.
 *   - Kernels overlap their predecessor on the stream (programmatic
 *     dependent launch): each may start before the kernel enqueued just
 *     before it has finished, and waits for it before touching anything
 *     that kernel may write.  kvring_write_frame reads its frame, and
 *     kvring_attention its queries, before that wait, except when a library
 *     kernel that may still be running writes a caller buffer overlapping
 *     them (kvring_project_write's q_out or kv_out, an attention output,
 *     the legacy window): the library records those buffers per stream and
 *     the call then reads after the wait.  A caller's own kernel launched
 *     with programmatic stream serialisation that triggers its dependents
 *     before it has written these inputs must not precede the library call
 *     that reads them.
 */
#ifndef KVRING_H
#define KVRING_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvring kvring_t;   /* opaque host handle, one per layer */

typedef enum {
  KVRING_OK = 0,
  KVRING_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size or config */
  KVRING_ERR_NOT_CALIBRATED = 2,  /* write or attention before calibration */
  KVRING_ERR_CAPACITY = 3,        /* more tokens than the ring or config allows */
  KVRING_ERR_UNSUPPORTED = 4,     /* head_dim or device not supported */
  KVRING_ERR_CUDA = 5             /* a CUDA runtime call or launch failed */
} kvring_status;

typedef struct {
  int32_t num_heads;      /* H >= 1 */
  int32_t head_dim;       /* d: 64 or 128 */
  int32_t capacity;       /* C ring slots, 1 .. 2^24 */
  int32_t max_tokens;     /* most tokens per write / calibration / attention call */
  int32_t max_position;   /* RoPE table rows: positions lie in [0, max_position) */
  int32_t max_kv_splits;  /* most key/value partitions one attention call may use (1..32) */
  int32_t attn_precision; /* 0 = automatic per tile; 1..4 = fixed precision level */
  int32_t pinned_prefix;  /* P, 0 .. capacity - 1: slots [0, P) keep the first P tokens ever
                             written and are never overwritten; later tokens cycle over the
                             other capacity - P slots.  0 = the plain ring.  (The pages give
                             5,788 = 7 x 757 + 489 slots and do not say whether a part is
                             never evicted; P = 489 reads the remainder as such a part.) */
  int32_t rope_pairs_t;   /* 0 = 1-D RoPE (one position per token).  Else the 3-D variant: of
                             the head_dim/2 rotation pairs, [0, T) turn with the frame index t,
                             [T, T + Y) with the row y and the rest with the column x, each
                             section a RoPE of its own (local pair j of a section of 2m dims
                             turns by coordinate * base^(-2j/(2m))).  T >= 8; T, Y and the
                             column pairs are multiples of 8.  Positions are then int32
                             [n][3] = (t, y, x), required by every call that takes them;
                             slot positions hold t, and a reset turns only the temporal
                             pairs.  (The pages give one position per token; a video model's
                             tokens have three coordinates.) */
  int32_t rope_pairs_y;   /* Y, the row pairs of the 3-D variant (0 with 1-D RoPE) */
  double rope_base;       /* RoPE base, e.g. 10000 */
} kvring_config;

#define KVRING_DELTA_TO_OLDEST (-1)
#define KVRING_OUT_F32 0
#define KVRING_OUT_BF16 1

/* Layout of the int32 state[] array returned by kvring_export(). */
#define KVRING_STATE_HEAD 0        /* next slot to be written */
#define KVRING_STATE_NVALID 1      /* filled slots: min(capacity, tokens written) */
#define KVRING_STATE_TOTAL_LO 2    /* tokens written, low 32 bits */
#define KVRING_STATE_TOTAL_HI 3    /* tokens written, high 32 bits */
#define KVRING_STATE_NEXT_POS 4    /* position given to the next token by default */
#define KVRING_STATE_CALIBRATED 5  /* 1 once scales are set */
#define KVRING_STATE_ERROR 6       /* device error bits, see KVRING_DEVERR_* */
#define KVRING_STATE_LAST_DELTA 7  /* delta used by the last delta rotation */
#define KVRING_STATE_WORDS 8

#define KVRING_DEVERR_POSITION 1u  /* a position outside [0, max_position) was skipped */
#define KVRING_DEVERR_TIMEOUT 2u   /* a pipeline wait in the attention kernel gave up */
#define KVRING_DEVERR_DELTA 4u     /* delta outside [0, max_position): rotation skipped */

/* Bytes of device memory one ring needs (cache, scales, positions, state,
 * RoPE table, attention workspace).  0 if the config is invalid. */
size_t kvring_required_bytes(const kvring_config* cfg);

/* Create a ring inside `dev_buf` (device memory of at least
 * kvring_required_bytes(cfg) bytes, 256-byte aligned, owned by the caller,
 * which must keep it alive until kvring_destroy and free it afterwards).
 * Clears the ring, uploads the RoPE table and builds the TMA descriptors.
 * This is the only call that synchronises (it waits for its own upload on
 * `stream`).  On success *out receives the handle. */
kvring_status kvring_create(const kvring_config* cfg, void* dev_buf, size_t bytes,
                            void* stream, kvring_t** out);

/* Free the host handle.  The device buffer stays the caller's. */
kvring_status kvring_destroy(kvring_t* ring);

/* Once per session ("Do It Once, at Write Time": per-head scales calibrated
 * once per session).  k, v: bf16 [n][H][d]; pos: int32 [n] device positions
 * of the keys, or NULL for next_pos + i (3-D RoPE: int32 [n][3], required).  For each head h:
 *   scale_k[h] = max |rope(k)[., h, .]| / 448, scale_v[h] = max |v[., h, .]| / 448
 * (IEEE single division; a result below 2^-126, e.g. an all-zero head,
 * becomes 1), and the reciprocals used for quantisation.  Writes nothing
 * into the ring; usually followed by kvring_write_frame of the same frame.
 * Errors: INVALID_ARG (n < 1, bad pointers), CAPACITY (n > max_tokens). */
kvring_status kvring_calibrate_scales(kvring_t* ring, const void* k_bf16, const void* v_bf16,
                                      const int32_t* pos, int32_t n, void* stream);

/* Write one frame of n new tokens ("Do It Once, at Write Time").
 * Token t goes to slot (head + t) mod capacity (with a pinned prefix P:
 * the g-th token ever written goes to slot g while g < P, else to slot
 * P + (g - P) mod (capacity - P)):
 *   K[h][slot][:] = e4m3(rope(k[t,h,:], pos[t]) * inv_scale_k[h])
 *   V[h][slot][:] = e4m3(v[t,h,:] * inv_scale_v[h])
 *   slot_pos[slot] = pos[t]
 * then head advances by n slots, n_valid = min(capacity, n_valid + n),
 * total += n, next_pos += n.  RoPE is computed in fp32 from the fp32
 * cos/sin table with every product and sum rounded separately.
 * pos: int32 [n] device positions, or NULL for next_pos + t (3-D RoPE:
 * int32 [n][3] = (t, y, x), required; slot_pos[slot] = t).
 * Errors: NOT_CALIBRATED, CAPACITY (n > capacity, n > capacity - P when
 * P > 0, or n > max_tokens), INVALID_ARG. */
kvring_status kvring_write_frame(kvring_t* ring, const void* k_bf16, const void* v_bf16,
                                 const int32_t* pos, int32_t n, void* stream);

/* Position reset ("Do It Once, at Write Time": one delta rotation of the
 * cached window at each reset).  Every filled slot's key is rotated by
 * -delta in place, in the FP8 code units (no rescaling): for each pair
 * (a, b) of decoded codes and the table row (c, s) of delta,
 *   a' = a*c + b*s,  b' = b*c - a*s   (fp32, each step rounded), then e4m3.
 * slot_pos -= delta for filled slots, next_pos -= delta.  Values are not
 * touched.  delta = KVRING_DELTA_TO_OLDEST reads, on the device, the
 * position of the oldest slot (the next slot to be overwritten once the
 * ring is full, slot 0 before), so the window restarts at position 0.
 * With a pinned prefix P only the rolling slots [P, n_valid) are rotated
 * and have their positions lowered (prefix keys are never re-rounded), and
 * KVRING_DELTA_TO_OLDEST takes delta = position of the oldest rolling slot -
 * (position of slot P - 1 + 1), at least 0, so the window continues right
 * after the prefix.
 * Errors: INVALID_ARG (delta < -1 or >= max_position). */
kvring_status kvring_delta_rotate(kvring_t* ring, int32_t delta, void* stream);

/* ------------------------------------------------------------------------
 * QKV projection with the cache write in its epilogue ("fused pre-attention
 * kernels", section "Judging Quality When Pixels Can't": the projection,
 * RoPE and FP8 quantisation in front of the attention, fused).
 *
 * y = x W^T for one frame: x bf16 [n][d_model] (the block's input rows), W
 * bf16 [3 * num_heads * head_dim][d_model] (a linear layer's weight: output
 * rows by input columns; rows [0, H*d) make the queries, [H*d, 2*H*d) the
 * keys, [2*H*d, 3*H*d) the values).  Summed in fp32 on the tensor cores and
 * rounded once to bf16 (the projection's output format); then
 *   - queries: stored to q_out bf16 [n][num_heads][head_dim] (NULL = not
 *     stored), what kvring_attention takes;
 *   - with KVRING_PROJECT_WRITE: keys and values written into the ring
 *     exactly as kvring_write_frame(k, v, pos, n) writes those bf16 values
 *     (same positions, slots, state advance, error word); needs a
 *     calibrated ring and n <= capacity - pinned_prefix;
 *   - with KVRING_PROJECT_STORE_KV: keys and values also stored to kv_out
 *     bf16 [2][n][num_heads][head_dim] (keys first), e.g. to calibrate a new
 *     session's scales from its first frame.
 * d_model is a multiple of 64 (at least 64); n <= max_tokens.  An fp32
 * tensor-core sum may round to a bf16 one step away from the exactly rounded
 * sum when that sum lies that close to a rounding midpoint.
 * ------------------------------------------------------------------------ */
#define KVRING_PROJECT_WRITE 1
#define KVRING_PROJECT_STORE_KV 2
kvring_status kvring_project_write(kvring_t* ring, const void* x, const void* w, int32_t d_model,
                                   const int32_t* pos, int32_t n, void* q_out, void* kv_out,
                                   int32_t flags, void* stream);

/* The cache upkeep the ring replaced, kept as the comparison path ("Where
 * the Time Went": before the ring, every attention call re-applied RoPE to
 * every cached key, re-quantised the cache to FP8 and shifted the window by
 * copying it).  The caller keeps the window of the last `capacity` tokens,
 * unrotated bf16 [capacity][H][d] in time order, in two buffer pairs and
 * alternates them: this call copies wk_in/wv_in shifted by the n new tokens
 * (the n oldest leave once the window is full) plus the frame k/v (bf16
 * [n][H][d]) into wk_out/wv_out, takes per-head scales from the whole new
 * window (amax of the rotated keys, of the values, over 448), and rewrites
 * the ring's FP8 cache from it: window slot i -> ring slot i, key rotated at
 * position base + i (base = position of the oldest token in the window,
 * positions counting the tokens given so far from 0), same pinned fp32 RoPE
 * and E4M3 conversion as kvring_write_frame.  Afterwards kvring_attention
 * reads the ring as usual.  Do not mix with kvring_write_frame on one ring.
 * Errors: INVALID_ARG (NULL, unaligned or aliased buffers), CAPACITY
 * (n > capacity or n > max_tokens), UNSUPPORTED (a ring with a pinned
 * prefix or 3-D RoPE: the original upkeep had neither). */
kvring_status kvring_legacy_upkeep(kvring_t* ring, const void* wk_in, const void* wv_in, void* wk_out,
                                   void* wv_out, const void* k_bf16, const void* v_bf16, int32_t n,
                                   void* stream);

/* Largest number of rings one batched call takes (a model's layers). */
#define KVRING_MAX_BATCH 64

/* kvring_write_frame on num_rings rings at once, in one launch: ring i gets
 * k_bf16[i], v_bf16[i] and pos[i] (pos may be NULL, or any pos[i] NULL, for
 * next_pos + t of that ring).  Every ring must have the same num_heads,
 * head_dim, capacity and pinned_prefix; n applies to all.  The result on each ring is
 * byte-for-byte that of kvring_write_frame.  The reset of the page
 * ("Do It Once, at Write Time") and the per-step upkeep touch every layer,
 * and one launch over all of them moves hundreds of megabytes instead of a
 * few per launch.  `rings`, `k_bf16`, `v_bf16` and `pos` are host arrays of
 * num_rings entries (the pointers in them are device pointers); rings must
 * be distinct.
 * Errors: INVALID_ARG (num_rings outside 1..KVRING_MAX_BATCH, a NULL or
 * repeated ring, mismatched shapes, unaligned pointers), NOT_CALIBRATED,
 * CAPACITY; nothing is launched on an error. */
kvring_status kvring_write_frames_many(kvring_t* const* rings, int32_t num_rings,
                                       const void* const* k_bf16, const void* const* v_bf16,
                                       const int32_t* const* pos, int32_t n, void* stream);

/* kvring_delta_rotate on num_rings rings of the same num_heads, head_dim,
 * capacity and pinned_prefix in one launch (delta, or KVRING_DELTA_TO_OLDEST read per ring on
 * the device).  Each ring ends byte-for-byte as after kvring_delta_rotate.
 * Errors: INVALID_ARG (as above, or delta < -1 or >= a ring's max_position);
 * nothing is launched on an error. */
kvring_status kvring_delta_rotate_many(kvring_t* const* rings, int32_t num_rings, int32_t delta,
                                       void* stream);

/* FP8 attention of n_q queries over the ring ("Where the Time Went";
 * "Blackwell and Beyond Four GPUs": FP8 attention with per-head scales).
 *   out[t,h,:] = sum_j softmax_j(rope(q[t,h,:], qpos[t]) . Kdeq[h,j,:] / sqrt(d)) Vdeq[h,j,:]
 * over the filled slots j, with Kdeq = code * scale_k[h], Vdeq = code *
 * scale_v[h].  Slot order does not matter: keys carry their rotation.
 * Queries are split into 1 to 4 FP8 terms with a per-row scale; the
 * probabilities multiply V in half precision (V widened exactly from its
 * E4M3 codes), as one f16 term at levels 1-3 and as two (the f16 value and
 * the f16 rounding of what it left) at level 4; products accumulate in fp32
 * on the tensor cores.  The level (1-4 query terms) is chosen per 128-query
 * tile from L = max|rotated q| * max|k| and V = max|v| of the head, unless
 * attn_precision fixes it: 4 when V > 128 or L*V > 4800, else 1 when L <= 4
 * and V <= 0.5, else 2 while L*V <= 435, else 3.
 * q: bf16 [n_q][H][d]; qpos: int32 [n_q] device positions (3-D RoPE:
 * int32 [n_q][3], required), or NULL for
 * next_pos - n_q + t (the positions of the last n_q tokens written with
 * default positions).  out: [n_q][H][d], fp32 (KVRING_OUT_F32) or bf16
 * (KVRING_OUT_BF16).  An empty ring gives zeros.
 * Errors: NOT_CALIBRATED, CAPACITY (n_q > max_tokens), INVALID_ARG. */
kvring_status kvring_attention(kvring_t* ring, const void* q_bf16, const int32_t* qpos,
                               int32_t n_q, void* out, int32_t out_dtype, void* stream);

/* Attention that allocates nothing, for callers that cannot hand the library
 * device memory.  Some callers cannot allocate device memory at all: a
 * plugin living inside a host program that owns the whole device memory
 * pool, or a real-time loop where an allocation would stall the device or
 * break its memory budget.  This entry point computes exactly what
 * kvring_attention computes, with the same arguments and errors, but its
 * scratch (the precision level chosen for each 128-query tile and head)
 * lives in a fixed 128 KiB static device array inside the library rather
 * than in the ring's buffer.  Every GPU that loads the library holds that
 * array until the process exits.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - The first call on a device looks up the array's device address
 *     (once per device, with that device current); make that first call
 *     before any stream capture.
 *   - The array is shared by every call: calls that overlap on the GPU
 *     (other streams, other rings) race and must be ordered by the caller.
 *     Nothing in it needs to start at zero (each call writes every level
 *     it uses before reading it).
 *   - It uses at most 8 key/value splits, which merge inside their
 *     thread-block cluster, so it needs no split partials.  A call with more
 *     than 32,768 (128-query tile, head) units, i.e. more than 4 bytes of
 *     levels per unit beyond 128 KiB, returns KVRING_ERR_CAPACITY.
 * The paper has no counterpart: this is a deployment variant. */
kvring_status kvring_attention_noalloc(kvring_t* ring, const void* q_bf16, const int32_t* qpos,
                                       int32_t n_q, void* out, int32_t out_dtype, void* stream);

/* Copy the ring out for inspection (tests, snapshots).  Any pointer may be
 * NULL to skip that part.  k_out, v_out: uint8 [H][capacity][d] codes;
 * scales: float [4H] = scale_k, scale_v, inv_scale_k, inv_scale_v;
 * slot_pos: int32 [capacity] (INT32_MIN = empty); state: int32
 * [KVRING_STATE_WORDS].  Destinations may be device or pinned host memory;
 * the copies are enqueued on `stream` (the caller synchronises). */
kvring_status kvring_export(kvring_t* ring, void* k_out, void* v_out, float* scales,
                            int32_t* slot_pos, int32_t* state, void* stream);

/* Test support, not part of the cache: encode n fp32 values to E4M3 codes
 * with the same conversion the kernels use (device pointers). */
kvring_status kvring_debug_encode_e4m3(const float* in, uint8_t* out, int64_t n, void* stream);

/* Measurement support: the fixed cost of kvring_write_frame for n tokens.
 * Launches a kernel with the write's grid, launch mode (a programmatic
 * dependent of the preceding kernel), wait, ring-state read, completion
 * ticket and state publication, but no data: nothing is read from the
 * frame, nothing written to the cache, and the ring state is rewritten with
 * its current values.  (The delta rotation's counterpart is
 * kvring_delta_rotate with delta 0, which moves no rows.)
 * Errors: INVALID_ARG, CAPACITY (as kvring_write_frame). */
kvring_status kvring_debug_write_floor(kvring_t* ring, int32_t n, void* stream);

/* Test support for the attention kernel's bounded waits.  Every wait in the
 * kernel gives up after limit_ns of wall time (default one second); a wait
 * that gives up sets KVRING_DEVERR_TIMEOUT in the ring's error word and the
 * kernel drains its copies and MMAs, frees its tensor memory and returns, so
 * the context stays usable.  With stall = 1 the kernel's first QK waits on a
 * barrier that nothing ever completes, so every following attention call on
 * this ring takes that path on purpose (its output is not the attention);
 * stall = 0 restores normal calls.  Host-side setting only: takes effect on
 * calls enqueued afterwards.
 * Errors: INVALID_ARG (limit_ns outside [1000, 6e10], stall not 0 or 1). */
kvring_status kvring_debug_set_attention_wait(kvring_t* ring, int64_t limit_ns, int32_t stall);

/* Test support for the attention's early query preparation.  With default
 * positions the kernel prepares its queries before waiting for the
 * preceding kernel, for the positions implied by a next-position hint that
 * every write leaves as it starts, and after the wait redoes the
 * preparation if the ring's next position turned out different.  With
 * wrong = 1 the guess of every following attention call on this ring is
 * off by max_position (so also outside the RoPE table, which must not be
 * reported), which exercises the redo; wrong = 0 restores normal calls.
 * Host-side setting only: takes effect on calls enqueued afterwards.
 * Errors: INVALID_ARG (wrong not 0 or 1). */
kvring_status kvring_debug_attention_guess(kvring_t* ring, int32_t wrong);

/* Test support: the precision level (1..4) each attention tile used in the
 * last kvring_attention call, int32 [ceil(n_q/128)][H], copied to `levels`
 * (device or pinned host) on `stream`. */
kvring_status kvring_debug_attention_levels(kvring_t* ring, int32_t* levels, void* stream);

/* Test support: how many kvring_write_frame and kvring_attention calls so
 * far (in this process, all rings and streams) found that the previous
 * library kernel on their stream may write their frame or queries, and so
 * read them only after waiting for it. */
int64_t kvring_debug_late_reads(void);

/* Static text for a status code. */
const char* kvring_status_string(kvring_status s);

#ifdef __cplusplus
}
#endif
#endif /* KVRING_H */
