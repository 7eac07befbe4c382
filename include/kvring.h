/*
 * kvring — a write-time FP8 ring KV cache for one GPU (sm_103a) and the
 * attention that reads it.
 *
 * Source: "Runway Characters: Serving a 57B Video Diffusion Transformer for
 * Real-Time Conversation" (arXiv:2611.05642):
 *   Introduction ("The model") and App. G  each cache holds global slots,
 *         written once per session, ahead of a window ring of latent frames;
 *   §4.1  a ring cache with a device-side write position;
 *   §4.2  RoPE applied once at write, and a delta rotation of the cached keys
 *         when positions reset;
 *   §4.3  K and V stored as float8_e4m3, queries quantised per call;
 *   App. G  cache update and position reset; every attention call reads all
 *         valid slots of its cache.
 *
 * Every call is asynchronous on the caller's CUDA stream, moves no data
 * between host and device (except the two documented debug calls), and can
 * be captured in a CUDA graph: the write position lives in device memory and
 * is advanced by the write kernel itself.
 *
 * Memory: the caller owns all device memory.  kvring_create carves one
 * caller-allocated device workspace (kvring_workspace_bytes bytes, 256-byte
 * aligned) into the ring state, the RoPE tables, the e4m3 code arrays, the
 * scale arrays, a per-head scale table (6 x H fp32) and the query scratch.  The handle itself owns host memory only; kvring_destroy
 * frees that and nothing else.
 *
 * Numbers and layouts:
 *   H = heads, D = head_dim, S = n_slots.
 *   bf16 inputs are row-major [n][H][D]; positions are int32 [n][n_axes].
 *   K codes and V codes are e4m3 [H][S][D]; K and V scales are fp32
 *   [H][S_pad] (S_pad = S rounded up to a multiple of 4); a (token, head)
 *   row's dequantised value is code * scale.
 *
 * Errors: every call returns KVRING_OK (0) or a negative status; arguments
 * are checked on the host before anything is enqueued.  Conditions only the
 * GPU can see (a position outside the RoPE table, attention over an empty
 * ring, a wait that exceeded its time limit) set bits in a device-side error
 * word that kvring_debug_state reads; the kernels never trap.  Non-finite
 * inputs are undefined behaviour.  A handle must not be used by two host
 * threads at once.
 */
#ifndef KVRING_H
#define KVRING_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvring kvring;           /* opaque host handle */
typedef struct CUstream_st* kvring_stream; /* a cudaStream_t; NULL = legacy default stream */

enum {
  KVRING_OK = 0,
  KVRING_ERR_INVALID_ARG = -1,  /* null pointer, bad size or configuration */
  KVRING_ERR_MISALIGNED = -2,   /* a pointer is not aligned as required */
  KVRING_ERR_UNSUPPORTED = -3,  /* shape outside the kernels' set (see kvring_config) */
  KVRING_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed; kvring_last_cuda_error says which */
  KVRING_ERR_WORKSPACE = -5,    /* workspace too small */
  KVRING_ERR_NO_DEVICE = -6,    /* no sm_100-family GPU is current */
  KVRING_ERR_SEQUENCE = -8      /* call out of order (global slots: once, before any window write;
                                   fixed scales: calibrate once, after a write, before any reset) */
};

enum { KVRING_SCALES_TOKEN = 0, KVRING_SCALES_STATIC = 1 };

/* bits of the device-side error word */
enum {
  KVRING_DEVERR_POS_RANGE = 1,  /* a position fell outside its axis's RoPE table (clamped) */
  KVRING_DEVERR_EMPTY = 2,      /* attention over a ring with no valid slot (output zeros) */
  KVRING_DEVERR_TIMEOUT = 4     /* a kernel gave up on a wait after its time limit */
};

enum { KVRING_OUT_BF16 = 0, KVRING_OUT_F32 = 1 };

/*
 * Cache geometry and RoPE layout.
 *   heads      1 .. 128 for head_dim 64, 1 .. 64 for head_dim 128
 *              (heads * head_dim / 16 <= 512: one thread block holds a
 *              token's heads)
 *   head_dim   64 or 128
 *   n_slots    1 .. 1<<20 ring slots
 *   n_axes     1 .. 3 RoPE axes; axis 0 is the temporal axis (the one the
 *              delta rotation of kvring_reset_positions turns)
 *   axis_dims  channels per axis, each even, summing to head_dim; axis a
 *              covers channels [o_a, o_a + axis_dims[a]) with o_a the sum of
 *              the earlier axes, and its pair j is channels (o_a+2j, o_a+2j+1)
 *   pos_min, pos_count
 *              the RoPE table of axis a covers integer positions
 *              pos_min[a] .. pos_min[a] + pos_count[a] - 1 (pos_count >= 1);
 *              positions outside it are clamped and flagged
 *              (KVRING_DEVERR_POS_RANGE)
 *   rope_base  the frequency base: omega_{a,j} = rope_base^(-2j/axis_dims[a])
 *   out_dtype  KVRING_OUT_BF16 or KVRING_OUT_F32 for kvring_attend's output
 *   max_queries  the largest n_q one kvring_attend call may pass, 1 .. 1<<20;
 *              the workspace holds that many rotated, e4m3-coded query rows
 *              (max_queries * H * D bytes + their fp32 scales) as per-call
 *              scratch, so two kvring_attend calls on one ring must not run
 *              at the same time (in stream order they may follow each other)
 *   n_global   0 .. n_slots-1 global slots (Introduction, "The model"; App. G:
 *              1,246 in the paper's caches).  Slots 0 .. n_global-1 hold the
 *              session's global tokens, written once by kvring_write_global
 *              and never rotated; the window ring is slots n_global ..
 *              n_slots-1 (W = n_slots - n_global of them).  0: the whole
 *              cache is the window ring.
 *   scale_mode KVRING_SCALES_TOKEN: one scale per (token, head) row, its
 *              absmax / 448, recomputed at write and at reset.
 *              KVRING_SCALES_STATIC: the paper's per-(cache, head) scales
 *              (§4.3, App. G): per token until kvring_calibrate, which fixes
 *              one K and one V scale per head from the maxima written so far
 *              times a margin; from then on writes use them and resets keep
 *              them, values beyond the range saturating.
 */
typedef struct {
  int32_t heads;
  int32_t head_dim;
  int32_t n_slots;
  int32_t n_axes;
  int32_t axis_dims[3];
  int32_t pos_min[3];
  int32_t pos_count[3];
  double rope_base;
  int32_t out_dtype;
  int32_t max_queries;
  int32_t n_global;
  int32_t scale_mode;
} kvring_config;

/* Bytes of device workspace kvring_create needs for this configuration
 * (0 if the configuration is invalid). */
size_t kvring_workspace_bytes(const kvring_config* cfg);

/*
 * Create a ring in the caller's device workspace (device pointer, 256-byte
 * aligned, at least kvring_workspace_bytes).  Enqueued on ``stream``: zeroes
 * the ring state (write position 0, no valid slot, error word 0) and the code
 * and scale arrays, and uploads the fp32 RoPE tables (cos and sin of
 * pos * omega_{a,j}, formed in fp64 and rounded once).  The workspace must
 * stay allocated until kvring_destroy.  Paper §4.1 (one allocation per cache,
 * device-side write position).
 */
int kvring_create(const kvring_config* cfg, void* workspace, size_t workspace_bytes, kvring_stream stream,
                  kvring** out);

/*
 * Write n_new tokens (ring_kv_write).  Paper §4.2 (RoPE at write), §4.3 (FP8
 * at write), §4.1 (ring slot at the device-side write position).
 *   k, v   device bf16 [n_new][H][D], 16-byte aligned; not modified
 *   pos    device int32 [n_new][n_axes], 4-byte aligned
 *   n_new  1 .. W (= n_slots - n_global)
 * For token i and head h: K is rotated by RoPE at pos[i] in fp32, V is not;
 * each (token, head) row of K and of V gets one fp32 scale amax/448 and e4m3
 * codes round-to-nearest-even(x * (448/amax)) saturated to +-448; they go to
 * slot n_global + (wp + i) mod W, where wp is the device-side write position.
 * Then, on the device, wp <- (wp + n_new) mod W and
 * n_valid <- min(n_valid + n_new, S).  With n_global > 0 the global slots
 * must have been written first (else KVRING_ERR_SEQUENCE).
 */
int kvring_write(kvring* r, const void* k, const void* v, const int32_t* pos, int32_t n_new,
                 kvring_stream stream);

/*
 * Write the session's n_global global tokens (ring_kv_write), once, before
 * the first kvring_write.  Introduction ("The model") and App. G: the global
 * slots are written once per session; a position reset does not move them.
 *   k, v, pos  as kvring_write, with n rows
 *   n          exactly n_global (else KVRING_ERR_INVALID_ARG, also when the
 *              ring has no global slots)
 * Same arithmetic as kvring_write; token i goes to slot i, and then, on the
 * device, n_valid <- n_global (wp stays 0).  A second call, or one after a
 * kvring_write, returns KVRING_ERR_SEQUENCE before anything is enqueued (the
 * order is checked on the host, in the order the calls are made).
 */
int kvring_write_global(kvring* r, const void* k, const void* v, const int32_t* pos, int32_t n,
                        kvring_stream stream);

/*
 * RMS norm of Q and K ahead of RoPE (paper §4.4 "Fused pre-attention" and
 * App. G: each block RMS-normalises the new tokens' Q and K, squaring in
 * fp32, before RoPE and the FP8 write).  Host-only: keeps the pointers; every
 * later kvring_write / kvring_write_global normalises K, and every later
 * kvring_attend(_noalloc) normalises Q, in the same kernels.
 *   gamma_q, gamma_k  device bf16 [H][D] weights (16-byte aligned), owned by
 *                     the caller and kept alive while in use; NULL turns
 *                     that norm off (both NULL: no norm, the default).  A
 *                     weight shared by all heads ([D]) must be expanded to
 *                     [H][D] by the caller: the kernels read H * D values.
 *   eps               > 0 and finite when a weight is given
 * The K norm belongs to a session: set it before the first write, since a
 * change later leaves normalised and raw keys side by side in the ring.  On a
 * calibrated KVRING_SCALES_STATIC ring (whose fixed K scales were taken from
 * the keys as they were then) a change of the K weights or of eps with K
 * weights set returns KVRING_ERR_SEQUENCE; the Q norm may change at any time.
 * Per (token, head) row x of D channels: S = sum x_d^2 (bf16 squares summed
 * in fp64, rounded once to fp32), ms = S / D, rstd = 1/sqrt(fl32(ms + eps))
 * correctly rounded, x_d <- bf16(fl32(fl32(x_d * rstd) * gamma_d)); RoPE and
 * quantisation then act on x.  V is not normalised.  A captured graph keeps
 * the weights that were set when it was captured.
 */
int kvring_set_qk_norm(kvring* r, const void* gamma_q, const void* gamma_k, float eps);

/*
 * Fix the per-head scales of a KVRING_SCALES_STATIC ring (paper §4.3 and
 * App. G: scales calibrated once per session from the amax of what the first
 * steps wrote, times a margin of 1.5).  Until this call the write kernel
 * quantises per (token, head) and records, per head, the largest |value| of
 * K (after RoPE) and of V it wrote.  This call, enqueued on ``stream``:
 *   a = fl32(margin * amax), scale = fl32(a / 448), inv = fl32(448 / a)
 *   (0 and 0 when a = 0), for K and for V of every head; then every valid
 *   slot's K and V rows are re-quantised from their dequantised values (code *
 *   scale, fp32) as e4m3_rn_satfinite(fl32(x * inv)) and their scale entries
 *   set to the head's scale.
 * Later writes quantise with these scales (values beyond 448 * scale
 * saturate) and resets keep them (rotated keys beyond the range saturate:
 * the paper's clamp).  Attention is unchanged: every slot's scale entry holds
 * its head's scale.  The ring's mode is read on the device, so a captured
 * write stays valid across the calibration.
 *   margin  > 0, finite (else KVRING_ERR_INVALID_ARG); the paper uses 1.5
 * KVRING_ERR_SEQUENCE, before anything is enqueued, unless the ring is
 * KVRING_SCALES_STATIC, not yet calibrated, and has been written to; a
 * kvring_reset_positions on such a ring before its calibration is refused
 * the same way.
 */
int kvring_calibrate(kvring* r, float margin, kvring_stream stream);

/*
 * Position reset by d (delta_rerotate).  Paper §4.2 and App. G: every cached
 * key moves from temporal position p to p - d; with RoPE angles affine in the
 * position, that is one rotation R(-d * omega_{0,j}) of each temporal-axis
 * pair.  Every valid window key row (slots n_global .. n_valid-1: the global
 * keys' positions do not depend on the window) is dequantised (code * scale,
 * fp32), its temporal pairs are rotated in fp32 by the fp32-rounded cos/sin
 * of -d * omega_{0,j} (formed in fp64 on the host), and the row is
 * re-quantised with a fresh absmax scale (on a calibrated
 * KVRING_SCALES_STATIC ring: with its head's fixed scale, saturating), in
 * place.  Values and global keys are not touched.  ``d`` is a
 * host value and is baked into a captured graph.  Callers pass positions
 * shifted by -d to later calls; the library keeps no position counter.
 */
int kvring_reset_positions(kvring* r, int32_t d, kvring_stream stream);

/*
 * The position reset of several rings in one launch (delta_rerotate): the
 * same as kvring_reset_positions(rings[i], d) for every i, in one kernel
 * launch per 32 rings instead of one per ring.  Paper App. G: at a reset the
 * window caches of all the model's blocks are re-rotated; §4.1: the caches of
 * all layers live in one allocation, each ring a slice of it (a caller that
 * creates n rings at offsets k * kvring_workspace_bytes(cfg) of one buffer
 * has that layout; every ring keeps its own state).
 *   rings  n handles, all on the current device, with the same head_dim,
 *          axis_dims[0] and rope_base (one rotation table serves them all;
 *          else KVRING_ERR_INVALID_ARG); heads, n_slots and n_global may
 *          differ.  A KVRING_SCALES_STATIC ring must be calibrated (else
 *          KVRING_ERR_SEQUENCE).  Nothing is enqueued if any check fails.
 *   n      >= 1
 */
int kvring_reset_positions_batch(kvring* const* rings, int32_t n, int32_t d, kvring_stream stream);

/*
 * Attention of n_q queries over every valid slot (fp8_ring_attn).  Paper §4.3
 * (queries quantised per call; attention reads the FP8 cache with per-token
 * scales) and App. G (all slots read).
 *   q      device bf16 [n_q][H][D], 16-byte aligned
 *   q_pos  device int32 [n_q][n_axes]
 *   n_q    1 .. max_queries
 *   out    device [n_q][H][D], bf16 or fp32 as configured, 16-byte aligned
 * Each query row is rotated by RoPE at q_pos (fp32) and quantised to e4m3
 * with its own scale (a first kernel writes these codes to the workspace's
 * query scratch); out = softmax(q.k / sqrt(D)) v over slots
 * 0 .. n_valid-1 with dequantised q, k and v, no mask.  Scores come from FP8
 * tensor-core products with fp32 accumulation; the softmax weights are
 * rounded to fp16 for the weighted sum of V, and the row sums that normalise
 * it are taken from the same fp16 weights (so their rounding cancels).
 */
int kvring_attend(kvring* r, const void* q, const int32_t* q_pos, int32_t n_q, void* out,
                  kvring_stream stream);

/*
 * kvring_attend_noalloc: kvring_attend with its per-call query scratch taken
 * from a fixed array inside the library instead of from the ring's workspace.
 * The Runway Characters paper has no counterpart to this call; it is an
 * addition for callers that cannot allocate device memory when they attend:
 * a serving loop that reserved all of its device memory at start-up (its
 * rings were sized with a small max_queries and cannot grow), or a real-time
 * path that must not call an allocator because cudaMalloc / cudaFree can
 * block, synchronise the device and take unbounded time.  This call
 * allocates nothing: no cudaMalloc / cudaFree, no memory pool, no library
 * that allocates (PyTorch's included), and it leaves the workspace's query
 * scratch untouched.
 *
 *   arguments, output and results: as kvring_attend, except that n_q is not
 *   bounded by the ring's max_queries but by the static scratch:
 *     round_up(n_q * H * D, 1024) + H * round_up(n_q, 4) * 4 + 8 * H
 *       <= KVRING_NOALLOC_SCRATCH_BYTES (8 MiB)
 *   (the query codes, their scales and two per-head factors of the
 *   attention), e.g. up to 2,647 queries at 24 heads x 128.  A larger
 *   request returns KVRING_ERR_SCRATCH_LIMIT before anything is enqueued.
 *
 * The scratch is one array per device for the whole process.  Calls that
 * can overlap in time on one device (two streams, two host threads, two
 * rings) share it and race: order them on one stream or with events.  Calls
 * on one stream are safe.  Nothing in the scratch has to start at zero:
 * each call's first kernel writes every query row and scale that its second
 * kernel reads, and rows past n_q come from the tensor copy's zero fill.
 *
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current, once per device); that
 * first call should come before any stream capture begins.  The address is
 * kept for the life of the process: after a cudaDeviceReset (which unloads
 * the library's device image) this call must not be used again.  The ring's
 * device must be the current device (else KVRING_ERR_INVALID_ARG).
 */
#define KVRING_NOALLOC_SCRATCH_BYTES (8u << 20)
enum { KVRING_ERR_SCRATCH_LIMIT = -7 /* request larger than kvring_attend_noalloc's static scratch */ };
int kvring_attend_noalloc(kvring* r, const void* q, const int32_t* q_pos, int32_t n_q, void* out,
                          kvring_stream stream);

/* Free the host handle (the workspace stays the caller's). NULL is allowed. */
int kvring_destroy(kvring* r);

/* Static description of a status code. */
const char* kvring_status_string(int status);

/* The last cudaError_t value seen by a call that returned KVRING_ERR_CUDA
 * on this host thread. */
int kvring_last_cuda_error(void);

/*
 * Device pointers into the workspace, for inspection (tests, tools):
 * K codes, V codes, K scales, V scales, the int32 state word array
 * {wp, n_valid, error, internal}, and S_pad.  Any out pointer may be NULL.
 */
int kvring_layout(const kvring* r, void** k_codes, void** v_codes, void** k_scales, void** v_scales,
                  void** state, int32_t* s_pad);

/*
 * DEBUG, SYNCHRONISING: wait for ``stream`` and copy the device state to
 * out3 = {wp, n_valid, error bits}.  Not for the hot path (it is the one
 * host<->device read the library offers).
 */
int kvring_debug_state(const kvring* r, kvring_stream stream, int32_t* out3);

/*
 * DEBUG: the kernels' bounded barrier wait, on its own.  One block of two
 * warps waits on a barrier that expects two arrivals; it gets one, or both
 * when ``complete`` is non-zero.  A wait that has not ended after limit_ns
 * nanoseconds (1 .. 1e10) gives up the way every wait in the library does: it
 * raises the block's abort flag, and the block records KVRING_DEVERR_TIMEOUT
 * and returns.  out2: device int64 [2] = {error bits (0 or
 * KVRING_DEVERR_TIMEOUT), nanoseconds the wait lasted}, 8-byte aligned.
 * Asynchronous on ``stream``; the device stays usable afterwards.
 */
int kvring_debug_wait_timeout(int64_t limit_ns, int32_t complete, int64_t* out2, kvring_stream stream);

/*
 * The quantiser of ring_kv_write applied to raw fp32 rows, for checking the
 * e4m3 cast bit for bit: x device fp32 [rows][d] (16-byte aligned, d a
 * multiple of 16, 16 .. 256) -> codes device u8 [rows][d], scales device fp32
 * [rows].  Asynchronous on ``stream``.
 */
int kvring_debug_quantize(const float* x, int64_t rows, int32_t d, uint8_t* codes, float* scales,
                          kvring_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* KVRING_H */
