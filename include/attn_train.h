/*
 * attn_train.h -- C ABI of the GB300 (sm_103a) fused training-attention
 * library: forward (O and LSE) and a deterministic backward (dQ, dK, dV)
 * for full, causal and EAGLE3 Training-Time-Test masks, with GQA.
 *
 * What the operations compute
 * ---------------------------
 * Forward (SpecForge long-context post, "EAGLE3 Training": attention(Q,K,V)
 * = softmax(Q K^T / sqrt(d_k)) V; CS336 README, "Flash Attention (Triton)":
 * the forward also keeps the per-row logsumexp L):
 *     S = scale * Q K^T (+ mask: invisible pairs are -inf)
 *     LSE[q] = ln sum_kv exp(S[q,kv]),  O = exp(S - LSE) V
 * Backward (HOT-Step flash-attn-training, section 1: the fused backward
 * emits dQ|dK|dV; CS336 README: P is recomputed from L):
 *     P = exp(S - LSE), dV = P^T dO, dP = dO V^T, Delta = rowsum(dO * O),
 *     dS = P * (dP - Delta), dQ = scale dS K, dK = scale dS^T Q.
 * GQA: q head h reads kv head h / (Hq / Hkv); dK and dV of a kv head are the
 * sum over its q heads, accumulated in ascending head order.
 * A query row that sees no key gets O = 0 and LSE = 0 (HOT-Step section 6,
 * trap 9); full, causal and TTT masks produce such rows only through the
 * per-batch key lengths, a window mask also through its extents.
 *
 * Masks (SpecForge post, "Flex Attention", eagle3 mask_mod):
 *   ATTN_MASK_FULL    every key visible (self- or cross-attention, Skv != Sq ok)
 *   ATTN_MASK_CAUSAL  key kv visible to query q iff kv <= q (top-left aligned)
 *   ATTN_MASK_TTT     TTT step t = ttt_step with Skv == (t+1)*Sq: K/V hold t+1
 *                     segments of Sq rows; query q sees segment-0 keys
 *                     kv <= q - t (the causal part shrinks one diagonal per
 *                     appended segment) plus key i*Sq + q of each appended
 *                     segment i = 1..t (one diagonal entry each).
 *   ATTN_MASK_WINDOW  the band q - window_left <= kv <= q + window_right (the
 *                     HOT-Step page's self-attention over a window, section 4);
 *                     (w, 0) is a causal sliding window, (w, w) a symmetric one.
 * Per-batch key lengths (the padding terms of the eagle3 mask_mod): with
 * seq_lengths set, keys kv >= seq_lengths[b] of batch entry b are invisible
 * (for TTT: segment-0 keys kv >= seq_lengths[b], and the suffix diagonals of
 * rows q >= seq_lengths[b]); their dK and dV are 0.
 * Additive mask (HOT-Step section 3: its ops accept an arbitrary additive mask
 * shaped [S_kv, S], or [S_kv, S, 1, B] with broadcast): with add_mask set, the scores of the pairs
 * the mask kind admits become scale * q.k + M[b][q][kv] (M = -inf hides the
 * pair); one M for all heads.  Not with ATTN_MASK_TTT.
 *
 * Layout and types
 * ----------------
 * Every Q/K/V/O/dO/dQ/dK/dV tensor is [B, H, S, D] with D contiguous
 * (stride 1) and arbitrary element strides for B, H and S (so BHSD and BSHD
 * both work).  Q, K, V and dO are bf16; O, dQ, dK and dV are bf16 or fp32 as
 * attn_problem.out_dtype says.  Pointers must be 16-byte aligned and every
 * stride times the element size a multiple of 16 bytes.  D is 16, 32, 64 or
 * 128.  LSE is fp32 contiguous [B, Hq, Sq].  Arithmetic: bf16 MMA operands,
 * fp32 accumulation and softmax.
 *
 * Ownership and streams
 * ---------------------
 * All tensor pointers are device pointers owned by the caller (except in the
 * host-memory step entry points below); the library allocates no device
 * memory and keeps no state between calls besides a device error word, cached
 * driver entry points and the host-step sessions a caller creates.  Work is enqueued on the
 * caller's stream (a cudaStream_t passed as void*, NULL = legacy default) and
 * the calls return before it finishes.  Outputs are overwritten, not
 * accumulated; summing gradients over TTT steps is the caller's job.
 *
 * Errors
 * ------
 * Every entry point validates its arguments on the host before it enqueues
 * anything and returns a status; there is no fallback path.  The message for
 * the last non-OK status of the calling thread is attn_train_last_error().
 * Device-side pipeline waits are bounded: a wait that runs out records an
 * error in a device word and the kernel returns; attn_train_device_status()
 * synchronizes the stream, reads and clears that word.  While the word is set,
 * further kernels of this library return without doing work.
 */
#ifndef ATTN_TRAIN_H
#define ATTN_TRAIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_MASK_FULL = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_TTT = 2,
  ATTN_MASK_WINDOW = 3
} attn_mask_kind;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = 1,        /* malformed arguments (null pointer, bad size) */
  ATTN_ERR_UNSUPPORTED = 2,    /* well-formed but not supported (head dim, mask) */
  ATTN_ERR_ALIGNMENT = 3,      /* pointer or stride breaks the 16-byte rule */
  ATTN_ERR_WORKSPACE = 4,      /* workspace missing or too small */
  ATTN_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed */
  ATTN_ERR_DEVICE_TIMEOUT = 6, /* a device-side wait ran out of budget */
  ATTN_ERR_DEVICE_CHECK = 7    /* a device-side check of a -DATTN_DEBUG build failed */
} attn_status;

/* A [B, H, S, D] tensor view: D has stride 1, the other strides are in
 * elements of the tensor's type. */
typedef struct {
  const void* ptr;
  int64_t stride_b, stride_h, stride_s;
} attn_tensor;

/* Element type of the outputs O, dQ, dK and dV (inputs are always bf16). */
typedef enum { ATTN_OUT_BF16 = 0, ATTN_OUT_F32 = 1 } attn_out_dtype;

/* Problem shape.  mask is an attn_mask_kind; ttt_step is t for ATTN_MASK_TTT
 * (ignored otherwise); scale <= 0 selects 1/sqrt(D); out_dtype is an
 * attn_out_dtype for O (forward output and backward input), dQ, dK and dV.
 * fp32 outputs avoid the bf16 rounding of large GQA gradient sums (a bf16
 * value of magnitude 8 is only good to 2^-5).  window_left / window_right are
 * the extents of ATTN_MASK_WINDOW (>= 0; must be 0 for the other masks).
 * seq_lengths: NULL, or a device array of B int32 key lengths (4-byte
 * aligned, read by the kernels; values are clamped to [0, Skv], to [0, Sq]
 * for TTT).  add_mask: NULL, or a device bf16 additive mask with element
 * (b, q, kv) at add_mask[b * add_mask_sb + q * add_mask_sq + kv]
 * (add_mask_sb = 0: one mask for every batch entry); 16-byte aligned, both
 * strides multiples of 8 elements, add_mask_sq >= Skv. */
typedef struct {
  int B, Hq, Hkv, Sq, Skv, D;
  int mask;
  int ttt_step;
  float scale;
  int out_dtype;
  int window_left, window_right;
  const int32_t* seq_lengths;
  const void* add_mask;
  int64_t add_mask_sb, add_mask_sq;
} attn_problem;

/* Whether the problem is supported.  Pure host check, no side effects.
 * Requires B, Hq, Hkv, Sq, Skv > 0, Hq % Hkv == 0, D in {16, 32, 64, 128},
 * a known mask, ttt_step >= 0 and Skv == (ttt_step + 1) * Sq for TTT,
 * window extents >= 0 for ATTN_MASK_WINDOW (0 otherwise), and a 4-byte
 * aligned seq_lengths pointer.  Size limits (ATTN_ERR_UNSUPPORTED beyond):
 * Sq, Skv < 2^30; every launch's grid within CUDA's limits (128-row tiles
 * and B*Hq*Sq / 16 row blocks below 2^31); with an additive mask
 * round8(Sq) <= 64 * 65535 and, for a per-batch mask, B <= 65535. */
attn_status attn_train_supports(const attn_problem* p);

/* Bytes of device workspace attn_train_bwd needs: the fp32 Delta row
 * statistic, B * Hq * Sq * 4 bytes rounded up to 256; for a TTT step t > 0
 * also the per-row weight and score gradient of each suffix diagonal,
 * 2 * B * Hq * Sq * t * 4 bytes (each part rounded up to 256).  Linear in S.
 * With an additive mask also its bf16 transpose for the dK/dV pass,
 * Bm * Skv * round8(Sq) * 2 bytes (Bm = 1 for a shared mask, else B): the
 * size of the mask itself. */
attn_status attn_train_workspace_size(const attn_problem* p, size_t* bytes);

/* Forward.  Inputs q [B,Hq,Sq,D], k and v [B,Hkv,Skv,D]; outputs o
 * [B,Hq,Sq,D] (bf16) and lse [B,Hq,Sq] (fp32, natural log).  Kernels: one
 * tcgen05 kernel (two 128-row query tiles per CTA).  Same as
 * attn_train_fwd_ws with no workspace. */
attn_status attn_train_fwd(const attn_problem* p, attn_tensor q, attn_tensor k, attn_tensor v,
                           attn_tensor o, float* lse, void* stream);

/* Bytes of device workspace attn_train_fwd_ws uses for this problem; 0 when
 * the forward does not split.  The split (a scheduling choice; the pages'
 * kernels launch one program per query block): when one CTA per pair of query
 * tiles would not fill a GB300's 152 multiprocessors (few batch
 * entries and heads, long rows), each pair's key tiles are cut into chunks, one
 * CTA per chunk writes its unnormalised partial O rows and their running max
 * and sum (fp32) into the workspace, and a merge pass combines the chunks in a
 * fixed order by log-sum-exp (CS336 README, "Flash Attention (Triton)": the
 * running max and normaliser of the online softmax) -- the same result up to
 * rounding, bitwise reproducible.  Never for the TTT mask.  A pure function of
 * the problem (no device needed). */
attn_status attn_train_fwd_workspace_size(const attn_problem* p, size_t* bytes);

/* Forward with a workspace: workspace NULL runs attn_train_fwd; otherwise it is
 * a device buffer of at least attn_train_fwd_workspace_size bytes (256-byte
 * aligned, contents ignored, ATTN_ERR_WORKSPACE when too small) and the forward
 * splits its key range when that size is non-zero.  Kernels: the tcgen05
 * forward and, when split, the merge pass. */
attn_status attn_train_fwd_ws(const attn_problem* p, attn_tensor q, attn_tensor k, attn_tensor v,
                              attn_tensor o, float* lse, void* workspace, size_t ws_bytes,
                              void* stream);

/* Backward.  Inputs q, k, v, o (the forward's output), dout [B,Hq,Sq,D] and
 * lse (the forward's); outputs dq [B,Hq,Sq,D], dk and dv [B,Hkv,Skv,D],
 * overwritten.  workspace: device buffer of at least attn_train_workspace_size
 * bytes, 256-byte aligned, contents ignored.  Fixed schedule, no atomics: the
 * result is bitwise identical across runs.  Kernels: Delta prep, dK/dV pass,
 * dQ pass, and for TTT the suffix-diagonal pass. */
attn_status attn_train_bwd(const attn_problem* p, attn_tensor q, attn_tensor k, attn_tensor v,
                           attn_tensor o, attn_tensor dout, const float* lse, attn_tensor dq,
                           attn_tensor dk, attn_tensor dv, void* workspace, size_t ws_bytes,
                           void* stream);

/* The kernels a problem runs, as one JSON object (NUL-terminated) in `buf`:
 * per pass the kernel instantiation (head dim and, for the attention kernels,
 * whether the general-mask, additive-mask and split forms are used), the rows
 * and keys a CTA or a tile covers, the grid size, the pipeline depths (K/V ring
 * entries, Q/dO stages) and the dynamic shared memory per CTA; the forward's
 * key-range split (it applies when attn_train_fwd_ws is given a workspace);
 * the TTT suffix pass and the mask transpose when the problem has them.  Pure
 * host function: it reports the plan the entry points follow for *p, for
 * logs and benchmark records.  `needed` (may be NULL) receives the size the
 * description takes, NUL included; a NULL or smaller `buf` returns
 * ATTN_ERR_INVALID (after setting `needed`).  Same problem checks as
 * attn_train_supports.  The pages have no counterpart: it is the record of the
 * resolved kernel variant, tile sizes and stage counts that the benchmark lines
 * carry. */
attn_status attn_train_describe(const attn_problem* p, char* buf, size_t buf_len, size_t* needed);

/* The backward's passes, for attn_train_bwd_passes. */
typedef enum {
  ATTN_BWD_PREP = 1,  /* Delta = rowsum(dO * O) into the workspace */
  ATTN_BWD_DKDV = 2,  /* dK, dV of the tiled keys (needs PREP's Delta) */
  ATTN_BWD_DQ = 4,    /* dQ incl. TTT suffix-diagonal terms (needs PREP's Delta) */
  ATTN_BWD_TTT = 8,   /* dK, dV of the TTT suffix keys (needs PREP's Delta) */
  ATTN_BWD_ALL = 15
} attn_bwd_pass;

/* Same arguments and checks as attn_train_bwd, but enqueues only the passes
 * set in `passes` (a mask of attn_bwd_pass), in the order PREP, DKDV, DQ,
 * TTT.  DKDV, DQ and TTT read the Delta that PREP wrote into the workspace
 * and are independent of each other, so a caller may run them on different
 * streams once PREP is done, or time them one by one.  ATTN_BWD_TTT is a
 * no-op unless the mask is TTT with ttt_step > 0. */
attn_status attn_train_bwd_passes(const attn_problem* p, unsigned passes, attn_tensor q,
                                  attn_tensor k, attn_tensor v, attn_tensor o, attn_tensor dout,
                                  const float* lse, attn_tensor dq, attn_tensor dk, attn_tensor dv,
                                  void* workspace, size_t ws_bytes, void* stream);

/* Backward without a caller-provided workspace.  The pages have no
 * counterpart for this entry point; it exists for callers that cannot
 * allocate device memory: code plugged into a host framework that owns all
 * device memory and hands an operator only its inputs and outputs (no
 * workspace hook), and code on a path where cudaMalloc's implicit device
 * synchronization is not acceptable.  Same arguments, checks, kernels and
 * results as attn_train_bwd minus the workspace pair; it allocates nothing
 * (no cudaMalloc, cudaFree or allocating library call).
 *
 * Its scratch -- the backward's whole workspace, attn_train_workspace_size
 * bytes: the fp32 Delta row statistic (B * Hq * Sq * 4 bytes), for a TTT step
 * t > 0 the suffix diagonals' weights and score gradients (2 * t * B * Hq *
 * Sq * 4 bytes more), with an additive mask its bf16 transpose -- lives in a
 * 4 MiB array compiled into the library as device memory, held by every GPU
 * that loads the library until the process exits.  Limit:
 * attn_train_workspace_size(p) <= 4 MiB (4,194,304 bytes), i.e. up to
 * 1,048,576 query rows B * Hq * Sq for the full, causal and window masks
 * without an additive mask, and about 1,048,576 / (1 + 2t) rows at TTT step t
 * (each part is rounded up to 256 bytes).  Larger problems return
 * ATTN_ERR_WORKSPACE with a message giving the bytes needed (use
 * attn_train_bwd then).
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call on a device shares the one array and each call
 * rewrites all the scratch it reads, so nothing needs clearing between
 * calls; but calls whose work overlaps on the GPU (different streams, no
 * ordering between them) race on it and must be serialized by the caller. */
attn_status attn_train_bwd_noalloc(const attn_problem* p, attn_tensor q, attn_tensor k,
                                   attn_tensor v, attn_tensor o, attn_tensor dout,
                                   const float* lse, attn_tensor dq, attn_tensor dk,
                                   attn_tensor dv, void* stream);

/* ---- steps from host memory --------------------------------------------
 *
 * attn_train_step_host runs the forward and the backward of one problem whose
 * inputs and outputs are HOST arrays: it copies q, k, v and dout to the
 * device, computes O, LSE, dQ, dK and dV with the same kernels as
 * attn_train_fwd and attn_train_bwd, and copies the five results back.  A
 * session (attn_train_host_session_*) does the same for a sequence of steps
 * of one problem and overlaps each step's copies with its neighbours' kernels.
 *
 * Host arrays are dense: q, dout, o, dq [B, Hq, Sq, D]; k, v, dk, dv
 * [B, Hkv, Skv, D]; lse [B, Hq, Sq] (fp32).  q, k, v, dout are bf16; o, dq,
 * dk, dv have the problem's out_dtype.  In these entry points the problem's
 * seq_lengths and add_mask are host pointers as well (add_mask keeps its
 * strides add_mask_sb / add_mask_sq; no alignment needed); both are copied in
 * with every step.  Pinned host memory (cudaHostAlloc / cudaHostRegister)
 * lets the copies run alongside the kernels; pageable memory works but
 * serializes them.
 *
 * arena: caller-owned device buffer of at least
 * attn_train_step_host_arena_size bytes (attn_train_host_session_arena_size
 * for a session with more slots), 256-byte aligned, contents ignored.  It
 * holds the slots of chunk buffers (two by default; see below), as many
 * copies of the key lengths and mask, and the backward's workspace; the
 * library allocates no device memory.
 *
 * Pipelining.  A step is one chunk (kv_heads_per_chunk <= 0: the whole
 * problem), or chunks of kv_heads_per_chunk kv heads (1 to Hkv, with their
 * Hq/Hkv query heads each) of one batch entry; GQA groups are independent
 * problems and contiguous slices of the host arrays.  Chunks take the
 * slots in turn, also across the steps of a session.  Per chunk, on three
 * streams: its inputs are copied in while the previous chunk computes; O and
 * LSE are copied out during its backward; the backward runs Delta prep and dQ
 * first, so that dQ is copied out while dK and dV are computed.  In a session
 * the next step's copy-in overlaps this step's kernels, so one chunk per step
 * is the fastest choice there; smaller chunks overlap more within a single
 * step at the price of fuller kernel tails.  No kernel mixes heads, so the
 * results equal those of attn_train_fwd + attn_train_bwd on the whole problem
 * bit for bit.
 *
 * Slots.  A slot holds the device copies of one chunk's inputs and outputs.
 * With n slots, chunk c's copy-in may start once chunk c - n has been
 * computed, and chunk c's kernels may start once chunk c - n has been copied
 * out: the copies can run up to n - 1 chunks ahead of (inputs) or behind
 * (outputs) the kernels.  Two slots suffice while the host link delivers at
 * a steady rate.  More slots let the kernels ride through pauses of the host
 * copies: on GB300 (Grace host) copies of a few hundred MB were measured to
 * stall for 20-80 ms about twice a second, in either direction, on one or
 * two streams; n slots absorb a pause of about (n - 1) chunks of compute,
 * and the copies then catch up at the rate by which they are faster than
 * the kernels.  Results do not depend on n.
 *
 * Streams.  Compute is enqueued on `stream`; the copies run on two streams of
 * the session.  The first step waits for the work already on `stream` (the
 * arena may still be in use); later steps do not, so their copy-in runs
 * during the previous step's compute.  Calls return once everything is
 * enqueued.  attn_train_host_session_join makes `stream` wait for every copy
 * enqueued so far: the host outputs are valid after a join followed by a
 * synchronization of `stream`, and the host inputs of a step may be changed
 * only then.  Validation happens before anything is enqueued. */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  void* o;
  float* lse;
  void* dq;
  void* dk;
  void* dv;
} attn_host_io;

typedef struct attn_host_session_s* attn_host_session;

/* Largest slot count of a host-memory session. */
#define ATTN_HOST_MAX_SLOTS 16

/* Arena bytes for this problem and chunk size (kv_heads_per_chunk <= 0: one
 * chunk for the whole step), with two slots. */
attn_status attn_train_step_host_arena_size(const attn_problem* p, int kv_heads_per_chunk,
                                            size_t* bytes);
/* The same for a session of `slots` slots (2 to ATTN_HOST_MAX_SLOTS; other
 * values return ATTN_ERR_INVALID).  Each slot adds the device copies of one
 * chunk's inputs and outputs and one copy of the key lengths and mask. */
attn_status attn_train_host_session_arena_size(const attn_problem* p, int kv_heads_per_chunk,
                                               int slots, size_t* bytes);

/* One step: create a session, enqueue the step, join `stream`, release the
 * session.  The outputs are valid once `stream` has been synchronized. */
attn_status attn_train_step_host(const attn_problem* p, const attn_host_io* io,
                                 int kv_heads_per_chunk, void* arena, size_t arena_bytes,
                                 void* stream);

/* A session over `arena` for steps of problem *p (copied; its host key
 * lengths and mask pointers are read at every step).  Creates two CUDA
 * streams and a few events (host objects; no device memory). */
attn_status attn_train_host_session_create(const attn_problem* p, int kv_heads_per_chunk,
                                           void* arena, size_t arena_bytes,
                                           attn_host_session* out);
/* A session with `slots` slots (2 to ATTN_HOST_MAX_SLOTS) over an arena of
 * at least attn_train_host_session_arena_size(p, kv_heads_per_chunk, slots)
 * bytes; attn_train_host_session_create is the two-slot form. */
attn_status attn_train_host_session_create_slots(const attn_problem* p, int kv_heads_per_chunk,
                                                 int slots, void* arena, size_t arena_bytes,
                                                 attn_host_session* out);
/* Enqueues one step (copy-in, forward, backward, copy-out).  Arguments are
 * checked before anything is enqueued; a failure after that (a CUDA error)
 * leaves the session unusable: later steps return ATTN_ERR_INVALID, and the
 * caller joins, synchronizes and destroys it. */
attn_status attn_train_host_session_step(attn_host_session s, const attn_host_io* io,
                                         void* stream);
/* Makes `stream` wait for every copy the session has enqueued so far. */
attn_status attn_train_host_session_join(attn_host_session s, void* stream);
/* Releases the session (work still in flight completes; the arena must stay
 * allocated until it has). */
attn_status attn_train_host_session_destroy(attn_host_session s);

/* Soft-target log-softmax loss (SpecForge long-context post, "In-place
 * Gradient Calculation": the EAGLE3 loss of one TTT step),
 *     loss = -(1/rows) sum_r mask[r] sum_v target[r, v] log_softmax(logits[r])_v
 * over `rows` positions (B * T) and a vocabulary of V entries.
 *
 * Forward.  logits and target: device fp32 [rows, V] with row strides
 * ld_logits, ld_target >= V (elements), 4-byte aligned; rows that all start
 * on 16-byte boundaries (strides multiples of 4, 16-byte aligned bases) are
 * read with 16-byte loads, others with 4-byte loads.
 * mask: device fp32 [rows], or NULL for all ones.  Outputs (device fp32, 4-byte
 * aligned): row_loss [rows] = -sum_v target log_softmax (before the mask),
 * row_lse [rows] = logsumexp of the row (the page's m + ln d), row_tsum [rows]
 * = sum_v target, and loss [1] = the mean (NULL: not computed).  One pass over
 * logits and target; fixed-order reductions (bitwise reproducible).
 * Kernels: one per-row pass and, for loss, one single-block mean. */
attn_status attn_train_logsoftmax_loss_fwd(int64_t rows, int64_t V, const float* logits,
                                           int64_t ld_logits, const float* target,
                                           int64_t ld_target, const float* mask,
                                           float* row_loss, float* row_lse, float* row_tsum,
                                           float* loss, void* stream);

/* Backward, in place: overwrites logits [rows, V] with dloss/dlogits times
 * grad_loss[0] (device fp32 scalar; NULL = 1):
 *     logits[r, v] <- -(grad_loss mask[r] / rows) (target[r, v]
 *                     - softmax(logits[r])_v row_tsum[r])
 * using row_lse and row_tsum from the forward on the same logits.  Masked rows
 * become 0.  Same layout rules as the forward.  One kernel. */
attn_status attn_train_logsoftmax_loss_bwd(int64_t rows, int64_t V, float* logits,
                                           int64_t ld_logits, const float* target,
                                           int64_t ld_target, const float* mask,
                                           const float* row_lse, const float* row_tsum,
                                           const float* grad_loss, void* stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* attn_train_last_error(void);

/* Synchronizes `stream`, then reads and clears the device error word of the
 * current device.  Returns ATTN_ERR_DEVICE_TIMEOUT if a kernel recorded a wait
 * that ran out of budget since the last call, ATTN_ERR_DEVICE_CHECK if a
 * device-side check of a library built with -DATTN_DEBUG failed (tile
 * coordinates outside a tensor, a work item or workspace slot that does not
 * exist; the message names the check's site). */
attn_status attn_train_device_status(void* stream);

/* Per-wait budget of the device-side pipeline waits, in nanoseconds (default
 * 2e9).  Host-side setting for kernels launched afterwards by this thread's
 * process; values < 1e6 are raised to 1e6. */
attn_status attn_train_set_wait_budget_ns(uint64_t ns);

/* ---- test-only entry points ------------------------------------------- */

/* Device evaluation of the mask as the kernels schedule it, through the same
 * tile-range and masking calls the kernels make.  bits: device buffer of
 * 6 * Sq * Skv bytes, six [Sq, Skv] planes of 0/1 = pair visited and not
 * masked: plane 0 the forward, plane 1 the dK/dV pass, plane 2 the dQ pass,
 * each in the form the kernels run for this problem (the one-sided form for
 * full, causal and TTT masks without key lengths or additive mask, else the
 * general form); planes 3-5 the same three passes in the general form.  TTT
 * suffix diagonals are included as the kernels address them.  tiles (may be
 * NULL): ceil(Sq/128) x ceil(kv_main/128) tile classes (0 empty, 1 partial,
 * 2 full) of the tiled part, kv_main = Sq for TTT else Skv.  Every plane must
 * equal the visibility predicate (SpecForge post, "Flex Attention",
 * eagle3 mask_mod).  With seq_lengths set: the view of batch entry 0. */
attn_status attn_train_mask_pattern(const attn_problem* p, uint8_t* bits, uint8_t* tiles,
                                    void* stream);

/* One-tile tcgen05 descriptor probe.  mode 0: c[128][128] = a[128][D] b[128][D]^T
 * (both operands K-major in shared memory); mode 1: c[128][D] = a[128][128]
 * b[128][D] (a in tensor memory, b MN-major in shared memory).  a, b: device
 * bf16 row-major; c: device fp32. */
attn_status attn_train_probe_mma(int mode, int D, const void* a, const void* b, float* c,
                                 void* stream);

/* Launches a kernel whose bounded wait can never be satisfied, with a 50 ms
 * budget; attn_train_device_status() must then return ATTN_ERR_DEVICE_TIMEOUT. */
attn_status attn_train_selftest_wait_timeout(void* stream);

/* In a library built with -DATTN_DEBUG: launches a kernel whose device-side
 * check fails on purpose (site 99, no memory access); attn_train_device_status()
 * must then return ATTN_ERR_DEVICE_CHECK.  In a normal build: returns
 * ATTN_ERR_UNSUPPORTED and launches nothing. */
attn_status attn_train_selftest_debug_check(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_TRAIN_H */
