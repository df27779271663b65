/*
 * attn.h -- C ABI of libattn.so: the fused exact-attention forward pass for
 * NVIDIA GB300 (sm_103a).
 *
 * Operation (one call):
 *   O[b,h,i,:] = sum_{j in A(i)} softmax_j(scale * Q[b,h,i,:] . K[b,h,j,:]) V[b,h,j,:]
 *   LSE[b,h,i] = ln sum_{j in A(i)} exp(scale * Q[b,h,i,:] . K[b,h,j,:])
 * computed tile by tile with a running row maximum and row sum, the division
 * by the row sum deferred to the end, so the Nq x Nk score matrix never
 * reaches device memory.
 *   - "Fused Self Attention" (AWS Neuron NKI tutorial), sections "Background"
 *     (S = Q K^T, R = softmax(S) V), "Fusion to Save SBUF Space" (one strip of
 *     query rows at a time) and "Softmax implementation" (row maximum, row
 *     sum, division delayed until after the product with V).
 *   - PhotoRoom / xformers memory-efficient attention post ("torch-permute"
 *     copy): Q and K are read in tiles with a running softmax, and only the
 *     end result is written to main GPU memory.
 *   - "Profiling in PyTorch" part 3, "Deconstructing Naive Attention": scores
 *     are scaled, masked positions are filled with -inf before the softmax;
 *     "Introducing Scaled Dot Product Attention": is_causal=True.
 *   - NATTEN issue #142 "circular windowed attention": 2-D neighbourhood
 *     attention (each query attends the keys between its window start and
 *     end), its circular "wrap" mode, and a float32 logsumexp output shaped
 *     like q without its last dimension.
 *
 * Allowed sets A(i):
 *   ATTN_MASK_NONE   every key j < Nk.
 *   ATTN_MASK_CAUSAL j <= i (top-left alignment, also when Nq != Nk).
 *   ATTN_MASK_CAUSAL_BR j <= i + (Nk - Nq) (bottom-right alignment: the queries
 *                    are the last Nq of Nk tokens). With Nq > Nk the first
 *                    Nq - Nk rows see no key: O = 0, LSE = -inf (and zero
 *                    gradients in attn_bwd).
 *   ATTN_MASK_NA2D   tokens are row-major on a grid_h x grid_w grid (Nq = Nk =
 *                    grid_h * grid_w); along each axis the window holds k
 *                    positions (k odd: `window` along the rows, `window_w`
 *                    along the columns, 0 = `window`). A clamped axis shifts a
 *                    full window inward at the borders, start = clamp(c - k/2,
 *                    0, G - k); a wrapped axis takes the positions (c + t)
 *                    mod G, t in [-k/2, k/2]. `wrap`: 0 = neither axis wraps,
 *                    1 = both, 2 = the rows only, 3 = the columns only. With
 *                    dilation dl > 1 (NATTEN's convention): a clamped axis
 *                    keeps the keys of c's residue class modulo dl and applies
 *                    the rule above to the index inside that class; a wrapped
 *                    axis takes (c + dl * t) mod G. k * dl <= the grid side of
 *                    its axis, unless k = 1. A 1 x N grid with window 1 along
 *                    the rows is 1-D neighbourhood attention.
 *   ATTN_MASK_NA3D   tokens are row-major on a grid_d x grid_h x grid_w
 *                    volume (depth slowest; Nq = Nk = the product, the grid
 *                    given explicitly); the key is allowed iff each of the
 *                    three axes allows it by the rule above. `window_d` is the
 *                    window along the depth (0 = `window`), `wrap_d` 1 wraps
 *                    the depth; `window`, `window_w`, `wrap` and `dilation`
 *                    as for NA2D (one dilation for all three axes). The
 *                    NATTEN issue's requester works on such volumes and wraps
 *                    some of their axes.
 *
 * Data layout (device memory, owned and allocated by the caller):
 *   q, o : bf16 [B, H, Nq, d]   k, v : bf16 [B, H, Nk, d]   (contiguous by
 *          default; attn_fwd_ex accepts element strides for b, h and n, the
 *          last dimension always contiguous, e.g. NATTEN's heads-last
 *          [B, X, Y, heads, d] layout without a permute)
 *   lse  : fp32 [B, H, Nq] contiguous, natural log; NULL = not written.
 *   d in {32, 64, 128}. Pointers 16-byte aligned; element strides multiples
 *   of 8 (16 bytes).
 *
 * Execution: every call only enqueues work on a CUDA stream (the one set by
 * attn_set_stream for the calling thread, or attn_params_ex.stream) and
 * returns; it launches exactly one kernel. The library keeps one lazily
 * allocated device status word per device, and for unmasked problems whose
 * work is split across CTAs (see attn_params_ex.schedule) a workspace for
 * partial results: the caller's (attn_params_ex.workspace) or else one per
 * device, allocated on first need and grown when a larger one is needed.
 * Calls that use the library's workspace must not overlap on the device
 * (e.g. on two streams at once); give each concurrent stream its own.
 * Device-side failures (a bounded wait that ran out) are reported by
 * attn_get_device_status() after the caller synchronises the stream.
 *
 * Errors: every entry point returns ATTN_OK (0) or one of the codes below;
 * argument checks happen on the host before any CUDA call, so an invalid call
 * touches no device state. attn_last_error() gives a one-line message for
 * the calling thread's last failure.
 *
 * Logging: with ATTN_LOG=1 in the environment, every forward launch writes one
 * line to stderr: the entry point, head dimension, mask and kernel variant,
 * shapes, the neighbourhood parameters and the schedule (whole tasks or split,
 * persistent grid size, tasks, K/V-tile units).
 */
#ifndef EXACT_ATTENTION_69_ATTN_H
#define EXACT_ATTENTION_69_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 6

typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_NA2D = 2,
  ATTN_MASK_NA3D = 3,
  ATTN_MASK_CAUSAL_BR = 4
} attn_mask_kind;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* sizes < 1, scale not finite or <= 0, even or
                                oversized window, wrap without NA2D, NA2D with
                                Nq != Nk or a non-square Nq and no grid, ... */
  ATTN_ERR_UNSUPPORTED = 2,  /* d not in {32,64,128} */
  ATTN_ERR_MISALIGNED = 3,   /* a pointer not 16-byte aligned, a stride not a
                                multiple of 8 elements */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed; the
                                message names it */
  ATTN_ERR_TIMEOUT = 5       /* a device-side wait ran past its bound; the
                                kernel stopped early, outputs are undefined */
} attn_status;

/* Full parameter block for attn_fwd_ex. Call attn_params_init first: it sets
 * every field to its default (contiguous strides, dilation 1, no extras). */
typedef struct attn_params_ex {
  const void* q;   /* bf16, see layout above */
  const void* k;
  const void* v;
  void* o;         /* bf16 output */
  float* lse;      /* fp32 [B,H,Nq] output, or NULL */
  int B, H, Nq, Nk, d;
  float scale;     /* > 0 and finite, typically 1/sqrt(d) */
  int mask_kind;   /* attn_mask_kind */
  int window;      /* NA2D, NA3D: odd window size along the rows (and the
                      columns / depth unless window_w / window_d is set);
                      others: must be 0 */
  int dilation;    /* NA2D, NA3D: key stride >= 1 along each axis; others: 1 */
  int wrap;        /* NA2D, NA3D: 0 = rows and columns clamp, 1 = both wrap,
                      2 = the rows wrap, 3 = the columns wrap; others: 0 */
  int grid_h, grid_w; /* NA2D, NA3D rows and columns; NA2D 0,0 = square grid
                         of side sqrt(Nq); NA3D: required */
  /* element strides of dims (b, h, n); all zero = contiguous [B,H,N,d] */
  int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3];
  void* stream;    /* cudaStream_t; NULL = the calling thread's stream */
  int num_ctas;    /* persistent CTAs; 0 = one per SM (smaller values are for tests) */
  uint64_t timeout_ns; /* bound on every device-side wait; 0 = 2 seconds */
  int inject;      /* test hook: 1 = the loader withholds one K tile so that
                      the kernel's bounded wait runs out (ATTN_ERR_TIMEOUT);
                      0 otherwise */
  void* ev_start;  /* optional cudaEvent_t recorded right before the kernel */
  void* ev_stop;   /* optional cudaEvent_t recorded right after the kernel */
  int schedule;    /* work split over the persistent CTAs: 0 = automatic,
                      1 = whole (batch, head, 256-query) tasks round robin,
                      2 = equal shares of K/V tiles, a task cut between CTAs
                          merged by its last part (ATTN_MASK_NONE only) */
  void* workspace; /* optional device buffer for schedule 2, zero-filled
                      before its first use (later calls leave it reusable);
                      NULL = the library's own */
  uint64_t workspace_bytes; /* size of `workspace` */
  int window_w;    /* NA2D, NA3D: odd window size along the columns; 0 =
                      `window`; others: must be 0 */
  int grid_d;      /* NA3D: depth of the volume (>= 1); others: must be 0 */
  int window_d;    /* NA3D: odd window size along the depth; 0 = `window`;
                      others: must be 0 */
  int wrap_d;      /* NA3D: 1 = the depth wraps, 0 = it clamps; others: 0 */
} attn_params_ex;

/* Fill *p with defaults (zero pointers and sizes, dilation 1, contiguous). */
void attn_params_init(attn_params_ex* p);

/*
 * attn_fwd: the fused forward pass over contiguous bf16 [B,H,N,d] tensors.
 * q,k,v,o are device pointers, lse a device pointer or NULL. For
 * ATTN_MASK_NA2D the token grid is square, side sqrt(Nq) (else
 * ATTN_ERR_INVALID_ARG); use attn_fwd_ex for other grids and layouts.
 * Returns an attn_status code. Asynchronous on the thread's stream.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int Nq, int Nk, int d, float scale,
             int mask_kind, int window, int dilation, int wrap);

/* attn_fwd with every option (strides, grid, stream, events, test hooks). */
int attn_fwd_ex(const attn_params_ex* p);

/* Set the CUDA stream (a cudaStream_t, NULL = legacy default stream) used by
 * the calling thread's later attn_fwd calls. Thread-local; always ATTN_OK. */
int attn_set_stream(void* stream);

/* Read and clear the current device's status words: the library's own (used
 * by attn_fwd, attn_fwd_ex, attn_bwd) and the one inside attn_fwd_noalloc's
 * fixed array. Allocates nothing (a word that does not exist yet reads as
 * zero). Call after synchronising the stream of the calls in question.
 * Returns ATTN_OK, ATTN_ERR_TIMEOUT, or ATTN_ERR_CUDA if a word could not be
 * read. If detail is not NULL it receives 4 words: code, role (0 loader, 1
 * MMA issuer, 2 softmax), KV tile index, CTA index of the first failure (the
 * library's own word first). */
int attn_get_device_status(uint32_t* detail);

/* Static one-line description of a status code. */
const char* attn_error_string(int code);

/* One-line message about the calling thread's last failing call ("" if none). */
const char* attn_last_error(void);

/* Number of SMs the persistent grid would use on the current device, or a
 * negative attn_status on failure. */
int attn_device_sm_count(void);

/* Bytes of workspace the call described by *p needs on the current device (0
 * if its schedule splits no task), or a negative attn_status. */
int64_t attn_workspace_bytes(const attn_params_ex* p);

/* Schedule tuning: the split-KV schedule's work split, chosen per problem by
 * measurement (the pages' kernels tune their tile configuration per problem;
 * here the tiles are fixed per head dimension and the schedule is tuned).
 * For the problem described by *p, times `iters` launches (>= 1) of each
 * candidate: whole (batch, head, 256-query) tasks over every SM, and, without
 * a mask, equal shares of K/V tiles over G CTAs for several G from the SM count
 * down to a quarter of it. Uses p's buffers (o and lse are overwritten) and
 * stream, and is synchronous. p->schedule and p->num_ctas are ignored; the
 * fastest candidate goes to *out, to be set in the params of later calls.
 * Returns an attn_status code. */
typedef struct attn_tune_result {
  int schedule;      /* 1 = whole tasks, 2 = equal K/V shares */
  int num_ctas;      /* persistent CTAs (0 = one per SM) */
  float us;          /* mean time per launch of that candidate */
  int n_tried;       /* candidates timed */
} attn_tune_result;

int attn_tune(const attn_params_ex* p, int iters, attn_tune_result* out);

/* Free the library's per-device state (status words, workspaces, the
 * backward's stream and scratch) and forget the no-alloc array's device
 * addresses. Later calls re-create it; the first attn_fwd_noalloc call on a
 * device after this looks the address up again, so it too must come before
 * any stream capture. */
void attn_shutdown(void);

/* ATTN_ABI_VERSION of the built library. */
int attn_abi_version(void);

/* sizeof(attn_params_ex) in the built library (lets bindings check their
 * copy of the struct layout). */
int attn_params_size(void);

/*
 * Backward pass: the gradients of a scalar loss through attn_fwd, given the
 * loss's gradient dout at the output O. With P the forward's softmax weights
 * (recomputed from Q, K and the saved log-sum-exp) and D_i = dout_i . O_i:
 *   dV = P^T dout,  dS = P * (dout V^T - D),  dQ = scale dS K,  dK = scale dS^T Q
 * (the chain rule through S = Q K^T, the row softmax and R = S V of "Fused Self
 * Attention", section "Background").
 * Layout: q, o, dout, dq: bf16 [B, H, Nq, d]; k, v, dk, dv: bf16 [B, H, Nk, d];
 * lse: fp32 [B, H, Nq] as written by attn_fwd; all contiguous, device memory
 * owned by the caller, 16-byte aligned. mask_kind and the neighbourhood
 * fields as for attn_fwd (the same checks apply). dq, dk and dv are
 * overwritten. Three kernels are enqueued: rowsum(dout * O) and dQ on the
 * stream, dK and dV on a library-owned second stream forked from it after the
 * first kernel and joined back into it (so later work on the stream, and CUDA
 * graph capture, see one ordered call). The library keeps a lazily grown
 * per-device scratch of B*H*Nq floats for D, so calls on one device must not
 * overlap in time.
 */
typedef struct attn_bwd_params {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int B, H, Nq, Nk, d;
  float scale;          /* the forward's scale */
  int mask_kind;        /* attn_mask_kind */
  void* stream;         /* cudaStream_t; NULL = the calling thread's stream */
  uint64_t timeout_ns;  /* bound on every device-side wait; 0 = 2 seconds */
  int window, window_w, dilation, wrap, grid_h, grid_w;  /* NA2D/NA3D, as attn_params_ex */
  int grid_d, window_d, wrap_d;                          /* NA3D, as attn_params_ex */
} attn_bwd_params;

/* Zero every field of *p, dilation 1. */
void attn_bwd_params_init(attn_bwd_params* p);

/* The backward pass; returns an attn_status code. Asynchronous. */
int attn_bwd(const attn_bwd_params* p);

/*
 * attn_fwd_noalloc: attn_fwd_ex for callers that cannot allocate device
 * memory -- code that runs where cudaMalloc is forbidden or unavailable (an
 * allocator's or memory pool's own internals, an embedded runtime that owns
 * every allocation) or that must never allocate lazily on a first call. The
 * pages describe no such entry point; it has no counterpart there.
 *
 * Computes the unmasked forward pass (mask_kind must be ATTN_MASK_NONE,
 * workspace NULL) with the split schedule, keeping every piece of scratch in
 * one fixed 48 MiB device array inside the library, which each GPU that loads
 * the library holds until the process exits. It calls no cudaMalloc,
 * cudaFree or other allocating routine. The caller passes inputs and outputs
 * as for attn_fwd_ex.
 *  - The first call on a device looks up the array's device address for that
 *    device (cudaGetSymbolAddress); make that first call before any stream
 *    capture.
 *  - A problem that needs more scratch than the array holds is rejected with
 *    ATTN_ERR_INVALID_ARG and a message giving both sizes.
 *  - All calls on a device share its array and each overwrites what the last
 *    one left. Calls that overlap on the GPU (e.g. on two streams at once)
 *    race and give wrong results: serialise them.
 *  - A device-side wait that runs out is recorded in the array's own status
 *    word; attn_get_device_status reads and clears it (allocating nothing).
 */
int attn_fwd_noalloc(const attn_params_ex* p);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_69_ATTN_H */
