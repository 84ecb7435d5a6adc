/*
 * gdn_decode.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet decode library.
 *
 * One decode step of a Gated DeltaNet (GDN) linear-attention layer, one token
 * a row, over slot-indexed state pools:
 *
 *   causal_conv1d_decode   depthwise width-W causal conv (+ SiLU) over the
 *                          packed q|k|v channels, rolling a per-slot conv
 *                          window.  "mstar PR #1139", section "What changed"
 *                          (the decode-only conv: the conv state update for one
 *                          token a row, with null slots, strided rows, optional
 *                          bias and activation, and a write slot).
 *   gdn_decode_step        the gated delta rule per row and value head:
 *                            alpha = exp(-exp(A_log) * softplus(a + dt_bias))
 *                            beta  = sigmoid(b)
 *                            q^ = q / sqrt(|q|^2 + 1e-6) / sqrt(dk)
 *                            k^ = k / sqrt(|k|^2 + 1e-6)
 *                            S' = alpha * S * (I - beta k^ k^T) + beta v k^T
 *                            o  = S' q^
 *                          "mstar PR #1139", section "Why" (the GDN rule, the
 *                          recurrent state update, is state traffic) and
 *                          "What changed" (twin slots: read one slot, write the
 *                          other, commit swaps them; in place for other walks).
 *   gdn_layer_decode       both of the above in one kernel.
 *   gdn_commit             the twin-slot commit (swap read and write slots).
 *
 * Conventions
 *  - Every function returns a status (GDN_OK = 0).  On failure a message is
 *    left in a thread-local buffer read by gdn_last_error().
 *  - Tensor arguments are DEVICE pointers unless stated otherwise; rows are
 *    contiguous and densely packed unless a row stride is given.  The caller
 *    owns every activation buffer.  Activation buffers (q, k, v, x, a, b and
 *    the outputs) may also be page-locked host memory mapped into the
 *    device's address space (cudaHostAlloc, or pinned memory under unified
 *    addressing): the kernels then read and write it across the host link,
 *    with no separate copy.  Pools, slot tables, taps, A_log and dt_bias are
 *    device memory, and so are gdn_prefill_chunked's activations.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Compute
 *    calls only enqueue work: no host synchronisation and no allocation.  The
 *    first call on a device looks up the library's device error word, so
 *    make one call on each device before capturing a CUDA graph.  Pool
 *    create/destroy and gdn_validate_slots / gdn_get_device_error synchronise.
 *  - Activation dtype: GDN_F32 or GDN_BF16 (q, k, v, a, b, x, conv weights and
 *    bias, conv pool, outputs).  The recurrent state is always fp32, and
 *    A_log and dt_bias are always fp32.
 *  - Slot 0 of every pool is the null slot.  A row whose read slot is 0 is a
 *    padding row: it reads and writes no slot and its outputs are written as
 *    zeros ("mstar PR #1127", "What changed": padding rows sit on slot 0,
 *    which stays zero; "mstar PR #965", "What changed": rows on the null slot
 *    change no real row's result).
 *  - Bad slots found on the device (a read or write slot outside
 *    [0, num_slots), a real row whose write slot is 0, or a twin row whose
 *    write slot equals its read slot) skip that row, zero its outputs and set
 *    a sticky per-device error word, read and cleared by
 *    gdn_get_device_error().  Kernels never trap or assert; every wait on a
 *    shared-memory barrier gives up one second after it began (the GPU's
 *    global timer) and reports GDN_DEVERR_TIMEOUT.
 *  - Scratch: the state kernels' two work counters live in the library's
 *    device memory (one pair a pool handle); gdn_prefill_chunked's
 *    workspace for bf16 activations is caller-owned device memory.
 *  - Preconditions not checked on the fast path: real rows name distinct
 *    write slots, and no row writes a slot another row reads.
 *    gdn_validate_slots() checks them (it synchronises).
 *  - Launches of gdn_decode_step / gdn_layer_decode that use the same state
 *    pool must not overlap on the GPU: issue them on one stream, or order
 *    them with events.  Each pool handle owns a pair of work counters that
 *    its launches share (the kernels hand out the tail of their work through
 *    them and leave them at zero when they end); overlapping launches on one
 *    pool race on that pair.  Launches on different pools may overlap.
 */
#ifndef GDN_DECODE_H
#define GDN_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define GDN_OK 0
#define GDN_EINVAL 1       /* bad argument: null pointer, bad size, bad dtype */
#define GDN_ENOMEM 2       /* device allocation failed (pool create only) */
#define GDN_ECUDA 3        /* a CUDA runtime call failed (message has details) */
#define GDN_EUNSUPPORTED 4 /* a shape the kernels are not built for */
#define GDN_ESLOTS 5       /* gdn_validate_slots found a violation */

/* ---- device error word values (gdn_get_device_error) ------------------ */
#define GDN_DEVERR_NONE 0
#define GDN_DEVERR_BAD_SLOT 1 /* some row named a slot outside the pool */
#define GDN_DEVERR_TIMEOUT 2  /* a bounded wait inside a kernel ran out; its CTA stopped */

/* ---- limits ------------------------------------------------------------ */
#define GDN_MAX_POOLS 4096 /* state pool handles alive at once, per process */

/* ---- activation dtypes ------------------------------------------------ */
#define GDN_F32 0
#define GDN_BF16 1

/* Head geometry of one GDN layer.  hv % hk == 0: value head h reads qk head
 * h / (hv / hk) (consecutive value heads share a qk head).  dk is one of
 * 16, 32, 64, 128, 256; dv is a multiple of 8, at most 512. */
typedef struct gdn_dims {
    int hk;
    int hv;
    int dk;
    int dv;
} gdn_dims;

typedef struct gdn_pool gdn_pool;   /* recurrent state pool (opaque) */
typedef struct conv_pool conv_pool; /* conv window pool (opaque) */

/* Message for the last failing call on this thread ("" if none). */
const char *gdn_last_error(void);

/* Library ABI version (increases when a signature changes). */
int gdn_abi_version(void);

/* ---- recurrent state pool -------------------------------------------- *
 * Layout: [num_slots][hv][dv][dk] fp32, dk contiguous; S[i][j] maps key
 * component j to value component i.  One slot is one request's state for
 * this layer; with twin slots a request holds two ("mstar PR #1139", "What
 * changed").  Slot 0 is the null slot.
 *
 * gdn_state_pool_create allocates and zero-fills (on `stream`, then waits
 * for it); the library owns the memory and frees it in
 * gdn_state_pool_destroy.  Returns GDN_ENOMEM when the device is full.
 * gdn_state_pool_wrap adopts caller memory (e.g. a torch tensor) of exactly
 * num_slots*hv*dv*dk floats, 16-byte aligned; it makes no CUDA call, and
 * destroy then frees only the handle.  num_slots >= 1.  Every handle also
 * takes one pair of work counters from a fixed table in the library's device
 * memory (GDN_MAX_POOLS pairs; GDN_ENOMEM once all are taken) and returns it
 * in gdn_state_pool_destroy, which must come after the pool's last launch has
 * finished.  gdn_state_pool_create also allocates the pool's in-place
 * counters (below); a wrapped pool has none until some are attached. */
int gdn_state_pool_create(int num_slots, gdn_dims dims, void *stream, gdn_pool **out);
int gdn_state_pool_wrap(void *dev_ptr, int num_slots, gdn_dims dims, gdn_pool **out);
int gdn_state_pool_destroy(gdn_pool *pool);

/* In-place counters: scheduling scratch of the fused layer in place
 * (gdn_layer_decode and its variants with keep_in_place), one 32-bit counter
 * per (slot, qk head), zero between launches.  A qk head's conv window is
 * read by the items of all its value heads and, in place ("mstar PR #1139",
 * "What changed": keep_in_place updates the slot a row reads), rewritten in
 * the same slot, so it must be written after its last read.  With the counters, a
 * launch spreads those items over all CTAs (as twin launches do) and the
 * item that counts last writes the window; without them each CTA takes
 * whole qk heads, which leaves most of the GPU idle below about 30 rows
 * (so do two shapes whose kept window does not fit beside the kernel's
 * ring: dk = 256 with width 3 in bf16 and with width 4 in fp32).  Results
 * are bit-identical either way.
 * gdn_pool_inplace_counter_bytes gives the size for a pool (0 for bad
 * arguments).  gdn_pool_attach_inplace_counters gives a wrapped pool
 * caller-owned device memory of at least that size, 16-byte aligned and
 * zero-filled, which must stay allocated while launches may use it; NULL
 * detaches them.  It makes no CUDA call; GDN_EINVAL for a pool made by
 * gdn_state_pool_create (it has its own), a NULL pool, a misaligned or short
 * buffer.  Counters are left set only by a launch that stopped on
 * GDN_DEVERR_TIMEOUT or by an in-place launch whose live rows name one slot
 * twice (a caller error: their states race); gdn_pool_zero_slots clears the
 * listed slots' counters with their states. */
size_t gdn_pool_inplace_counter_bytes(int num_slots, gdn_dims dims);
int gdn_pool_attach_inplace_counters(gdn_pool *pool, void *dev_counters, size_t bytes);
void *gdn_pool_data(const gdn_pool *pool);
int gdn_pool_num_slots(const gdn_pool *pool);
gdn_dims gdn_pool_dims(const gdn_pool *pool);

/* Zero the n slots listed in the device array `slots` (a request's release
 * or rollback zeroes both of its slots: "mstar PR #1139", "Tests"), and
 * their in-place counters if the pool has them.  Slots outside
 * [0, num_slots) are skipped and set the device error word.  n may be 0. */
int gdn_pool_zero_slots(gdn_pool *pool, const int32_t *slots, int n, void *stream);

/* Snapshots and forks: slot dst[i] receives an exact copy of slot src[i], for
 * i < n (src, dst: device int32 arrays).  A prefix-cache checkpoint copies a
 * request's state and conv window into snapshot slots, and a fork copies
 * them into a new request's slots ("mstar PR #1139", "What changed": prefix
 * snapshots of the conv window and state; "mstar PR #965", "What changed":
 * prefix-cache checkpoints).  A source outside [0, num_slots) or a
 * destination outside [1, num_slots) skips the pair and sets the device
 * error word (the null slot is never written).  Destinations must be
 * distinct and must not be sources.  n may be 0.  conv_pool_copy_slots does
 * the same for a conv pool. */
int gdn_pool_copy_slots(gdn_pool *pool, const int32_t *src, const int32_t *dst, int n, void *stream);

/* ---- conv window pool ------------------------------------------------- *
 * Layout: [num_slots][width-1][channels] in the activation dtype, channel
 * contiguous, oldest input first.  width is 2..4; channels a multiple of 8.
 * Create/wrap/destroy/zero as for the state pool (wrap needs 16-byte
 * alignment). */
int conv_state_pool_create(int num_slots, int channels, int width, int dtype, void *stream,
                           conv_pool **out);
int conv_state_pool_wrap(void *dev_ptr, int num_slots, int channels, int width, int dtype,
                         conv_pool **out);
int conv_state_pool_destroy(conv_pool *pool);
void *conv_pool_data(const conv_pool *pool);
int conv_pool_num_slots(const conv_pool *pool);
int conv_pool_zero_slots(conv_pool *pool, const int32_t *slots, int n, void *stream);
int conv_pool_copy_slots(conv_pool *pool, const int32_t *src, const int32_t *dst, int n, void *stream);

/* ---- causal_conv1d_decode --------------------------------------------- *
 * For each row r with s = slot_idx[r] != 0 and each channel c:
 *   pre      = bias[c] + sum_{j<W-1} w[c][j] * win_s[j][c] + w[c][W-1] * x[r][c]
 *   out[r][c]= silu ? pre / (1 + exp(-pre)) : pre        (fp32, rounded once)
 *   window of write_slot[r] (or of s when write_slot == NULL) = [win_s[1..], x[r]]
 * Rows with slot 0 write out[r] = 0 and touch no slot.
 *   x          [rows] x channels, row stride x_row_stride elements (>= channels,
 *              multiple of 8); x, w, bias and out 16-byte aligned
 *   w          [channels][W];  bias [channels] or NULL
 *   out        [rows][channels], dense
 *   slot_idx   [rows] int32 read slots;  write_slot [rows] int32 or NULL
 * "mstar PR #1139", "What changed" and "Tests" (null slots, strided rows, no
 * bias or activation, a write slot leaving the read slot alone). */
int causal_conv1d_decode(const void *x, int x_row_stride, conv_pool *cp, const int32_t *slot_idx,
                         const int32_t *write_slot, const void *w, const void *bias, int silu,
                         void *out, int rows, int dtype, void *stream);

/* ---- gdn_decode_step --------------------------------------------------- *
 *   q, k   [rows][hk][dk]     v, out [rows][hv][dv]     a, b [rows][hv]
 *   A_log, dt_bias [hv] fp32
 *   read_slot [rows] int32; write_slot [rows] int32 (ignored when
 *   keep_in_place != 0, and may then be NULL)
 *   q, k and v are copied by the bulk-copy engine: each must be 16-byte
 *   aligned (GDN_EINVAL otherwise). 
 * For every real row and value head: S = pool[read_slot[r]][h]; the updated
 * state goes to write_slot[r] (twin) or back to read_slot[r] (in place); out
 * receives o.  `heads` must equal the pool's hv.  Twin and in-place calls
 * produce bit-identical values ("mstar PR #1139", "What changed": same
 * kernel, same values). */
int gdn_decode_step(const void *q, const void *k, const void *v, const void *a, const void *b,
                    const float *A_log, const float *dt_bias, gdn_pool *pool,
                    const int32_t *read_slot, const int32_t *write_slot, void *out, int rows,
                    int heads, int keep_in_place, int dtype, void *stream);

/* ---- gdn_layer_decode -------------------------------------------------- *
 * causal_conv1d_decode (SiLU on when silu != 0) followed by gdn_decode_step,
 * in one kernel.  The pages run the two as separate kernels ("mstar PR
 * #1139", "What changed": the decode conv as a kernel of its own beside the
 * GDN decode wrapper); this fusion is the library's own, with the same
 * values as the pair.  x is [rows][C], C = 2*hk*dk + hv*dv packed [q | k | v],
 * head-major; the conv pool must have C channels.  Both pools use the same
 * read/write slots.  The conv output is rounded to the activation dtype
 * before the rule, exactly as between the two separate calls, so the result
 * is bit-identical to causal_conv1d_decode + gdn_decode_step.  x, w and bias
 * must be 16-byte aligned. */
int gdn_layer_decode(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                     const float *A_log, const float *dt_bias, const void *a, const void *b,
                     gdn_pool *pool, const int32_t *read_slot, const int32_t *write_slot,
                     void *out, int rows, int keep_in_place, int dtype, void *stream);

/* ---- many tokens a sequence -------------------------------------------- *
 * Packed sequences: sequence r holds tokens [cu_seqlens[r], cu_seqlens[r+1])
 * of the token-major inputs (cu_seqlens [nseq+1] int32 on the device,
 * cu_seqlens[0] = 0, non-decreasing, cu_seqlens[nseq] = total_tokens; a
 * range outside [0, total_tokens] makes the sequence bad).  read_slot,
 * write_slot [nseq]; token_slot [total_tokens].  A sequence whose read slot
 * is 0 is padding (outputs zero, no slot touched); bad slots skip the
 * sequence, zero its outputs and set the device error word.
 *
 * gdn_prefill: the rule applied token after token, from the state in
 * read_slot[r]; the final state goes to write_slot[r] (twin) or back to
 * read_slot[r] (keep_in_place != 0, write_slot may be NULL).  ("mstar PR
 * #1139", "Why": the rule is the recurrent state update of one token, and
 * prefill keeps the state in place.)  Each token's output and every state
 * equal, bit for bit, the same tokens fed one decode step at a time
 * (gdn_decode_step, in place or twin).
 *   q, k [T][hk][dk]   v, out [T][hv][dv]   a, b [T][hv]   A_log, dt_bias [hv]
 *   q, k and v are bulk-copied: 16-byte aligned.
 * gdn_verify: as gdn_prefill, but the state after token t goes to
 * token_slot[t] and the read slot is left alone: a state a token, for
 * speculative decoding ("mstar PR #1139", "What changed": speculative
 * decoding holds a state per token).  Token slots must be real slots other
 * than the sequence's read slot.
 * causal_conv1d_prefill: the conv over a sequence, continuing the window in
 * read_slot[r]: x, out [T][C] (rows packed, C the pool's channels); the
 * window after the last token goes to write_slot[r] (NULL: in place), or,
 * when token_slot is given, the window after token t goes to token_slot[t].
 * Each token's output equals one causal_conv1d_decode call.  x, w, bias and
 * out 16-byte aligned. */
int gdn_prefill(const void *q, const void *k, const void *v, const void *a, const void *b,
                const float *A_log, const float *dt_bias, gdn_pool *pool, const int32_t *cu_seqlens,
                const int32_t *read_slot, const int32_t *write_slot, void *out, int nseq, int total_tokens,
                int keep_in_place, int dtype, void *stream);
/* gdn_prefill_chunked: gdn_prefill's operation and contract (same
 * arguments, slots, padding, bad sequences, in place or twin), computed in
 * chunks of 64 tokens on the tensor cores: the chunked GDN path that the
 * pages check the mixed step against ("mstar PR #965", "Correctness") and
 * run as one GDN prefill kernel ("mstar PR #1127").  Each product splits its
 * fp32 operands into bf16 heads and tails, so outputs and final states agree
 * with gdn_prefill to about 1e-5 relative per chunk, not bit for bit.  Built
 * for dk = dv = 128 (GDN_EUNSUPPORTED otherwise).  q, k, v 16-byte aligned.
 * bf16 activations run two kernels: every chunk's state-free terms (gates,
 * norms, P, T) in parallel into `workspace`, then the chunks of each
 * sequence in order.  The caller owns the workspace: device memory, 128-byte
 * aligned, at least gdn_prefill_chunked_workspace_bytes(nseq, total_tokens,
 * hv) bytes (GDN_EINVAL otherwise); its contents need no initialisation and
 * are garbage afterwards; calls that overlap on the GPU need their own.
 * fp32 activations ignore it (NULL allowed).  The bf16 call also encodes
 * three tensor maps (q, k, v) on the host for the chunk kernel's tensor
 * copies; should the driver refuse one, the call returns GDN_ECUDA and
 * launches nothing.  `out` needs no alignment beyond its element.
 * cu_seqlens must be nondecreasing: a sequence whose chunks the prep kernel
 * could not place counts as bad (zero outputs, GDN_DEVERR_BAD_SLOT, no
 * state written). */
size_t gdn_prefill_chunked_workspace_bytes(int nseq, int total_tokens, int hv);
int gdn_prefill_chunked(const void *q, const void *k, const void *v, const void *a, const void *b,
                        const float *A_log, const float *dt_bias, gdn_pool *pool, const int32_t *cu_seqlens,
                        const int32_t *read_slot, const int32_t *write_slot, void *out, int nseq,
                        int total_tokens, int keep_in_place, void *workspace, size_t workspace_bytes,
                        int dtype, void *stream);
int gdn_verify(const void *q, const void *k, const void *v, const void *a, const void *b,
               const float *A_log, const float *dt_bias, gdn_pool *pool, const int32_t *cu_seqlens,
               const int32_t *read_slot, const int32_t *token_slot, void *out, int nseq, int total_tokens,
               int dtype, void *stream);
int causal_conv1d_prefill(const void *x, conv_pool *cp, const int32_t *cu_seqlens, const int32_t *read_slot,
                          const int32_t *write_slot, const int32_t *token_slot, const void *w,
                          const void *bias, int silu, void *out, int nseq, int total_tokens, int dtype,
                          void *stream);

/* ---- gdn_layer_decode_commit ------------------------------------------- *
 * gdn_layer_decode in twin mode followed by gdn_commit, in one launch: the
 * same values, then read_slot[r] and write_slot[r] swapped for every row
 * ("mstar PR #1139", "What changed": twin slots, the commit swaps them).  For
 * the last layer of a step whose layers share one slot table; the kernel
 * swaps the tables once no CTA of the launch reads them any more, so the next
 * launch on the stream sees the committed tables. */
int gdn_layer_decode_commit(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                            const float *A_log, const float *dt_bias, const void *a, const void *b,
                            gdn_pool *pool, int32_t *read_slot, int32_t *write_slot, void *out,
                            int rows, int dtype, void *stream);

/* ---- gdn_layer_decode_bucket ------------------------------------------- *
 * The decode half of a mixed step ("mstar PR #965", "What changed": decode
 * rows lead the bucket, the GDN decode kernel runs over the leading run of
 * one-token rows, sized to the bucket, and the width changes no real row's
 * result).  The launch covers `rows` (the bucket); only rows below *n_decode
 * (an int32 on the device, read when the kernel runs, so a captured launch
 * can serve every decode count) are decoded, exactly as gdn_layer_decode
 * would decode them.  Rows at or past *n_decode are left alone: their outputs
 * are zero, and their slots, conv windows and table entries are not touched
 * even when they name real slots (they belong to the bucket's prefill rows).
 * With commit != 0 (twin only) the tables of the decoded rows are swapped in
 * the same launch, as by gdn_layer_decode_commit. */
int gdn_layer_decode_bucket(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                            const float *A_log, const float *dt_bias, const void *a, const void *b,
                            gdn_pool *pool, int32_t *read_slot, int32_t *write_slot, void *out, int rows,
                            const int32_t *n_decode, int keep_in_place, int commit, int dtype, void *stream);

/* ---- gdn_layer_decode_noalloc ------------------------------------------ *
 * gdn_layer_decode for callers that cannot allocate device memory; the pages
 * have no counterpart (it is an interface matter, not part of the method).
 * Such callers are, for example, engines that reserve all device memory up
 * front for their own allocator and forbid cudaMalloc elsewhere, and paths
 * where cudaMalloc's implicit device-wide synchronisation would stall other
 * streams.
 * Same arguments, checks and results, bit for bit, as gdn_layer_decode, plus
 * scratch_slot.  The call allocates nothing (no cudaMalloc, no allocating
 * library routine): the kernel's scratch, two 32-bit work counters, is slot
 * `scratch_slot` of a fixed array in the library's device memory of
 * GDN_NOALLOC_SCRATCH_SLOTS slots (8 bytes each, 512 bytes in all), whose
 * device address is looked up by the first call on each device (with that
 * device current; make that first call before any stream capture) and then
 * cached for the life of the process: it does not survive cudaDeviceReset
 * or a new primary context on that device, after which the call must not be
 * used again in the process.  A slot outside
 * [0, GDN_NOALLOC_SCRATCH_SLOTS) is rejected with GDN_EINVAL.  Both counters
 * of the slot must be zero when a launch starts: the array is zero when the
 * library loads and every launch leaves its slot at zero when it ends.
 * Calls that overlap on the GPU and use the same scratch slot race on it and
 * give wrong results; give concurrent calls different slots.  The state
 * pool's own work counters are not used by this call. */
#define GDN_NOALLOC_SCRATCH_SLOTS 64
int gdn_layer_decode_noalloc(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                             const float *A_log, const float *dt_bias, const void *a, const void *b,
                             gdn_pool *pool, const int32_t *read_slot, const int32_t *write_slot,
                             void *out, int rows, int keep_in_place, int scratch_slot, int dtype,
                             void *stream);

/* ---- gdn_commit -------------------------------------------------------- *
 * Twin-slot commit: swap read_slot[r] and write_slot[r] for every row, on the
 * device ("mstar PR #1139", "What changed": commit swaps them). */
int gdn_commit(int32_t *read_slot, int32_t *write_slot, int rows, void *stream);

/* ---- debugging --------------------------------------------------------- *
 * gdn_validate_slots copies the tables to the host (synchronising `stream`)
 * and returns GDN_ESLOTS with a message if a slot is out of range, a real
 * row writes the null slot, two real rows read or write one slot, a twin row
 * writes its own read slot, or a row writes a slot another row reads.
 * write_slot may be NULL when keep_in_place != 0. */
int gdn_validate_slots(const int32_t *read_slot, const int32_t *write_slot, int rows,
                       int num_slots, int keep_in_place, void *stream);

/* Synchronise `stream`, return the current device's error word in *code and
 * clear it. */
int gdn_get_device_error(int *code, void *stream);

/* Exercise the bounded-wait failure path: one thread waits, through the
 * same bounded wait the kernels use, on a shared-memory barrier that nothing
 * arrives at, giving up after `limit_us` microseconds (the kernels' waits give
 * up after one second).  The device error word then reads GDN_DEVERR_TIMEOUT;
 * nothing faults, no copy is left in flight, and the context serves the next
 * call.  Asynchronous on `stream`.  limit_us outside [1, 10^6] -> GDN_EINVAL. */
int gdn_selftest_wait_timeout(int limit_us, void *stream);

/* ---- roofline probes --------------------------------------------------- *
 * Move the state bytes of a step with no arithmetic, over the same pool
 * geometry and slot tables ("mstar PR #1139", "Numbers": the same reads and
 * writes with no math; read-only plus write-only).  mode:
 *   GDN_PROBE_TWIN     read the read slot, write the write slot
 *   GDN_PROBE_INPLACE  read and write back the read slot
 *   GDN_PROBE_READ     read only (sink may be NULL; it only keeps the loads
 *                      alive and is practically never written)
 *   GDN_PROBE_WRITE    write only (the write slot receives zeros) */
#define GDN_PROBE_TWIN 0
#define GDN_PROBE_INPLACE 1
#define GDN_PROBE_READ 2
#define GDN_PROBE_WRITE 3
int gdn_probe_traffic(gdn_pool *pool, const int32_t *read_slot, const int32_t *write_slot,
                      int rows, int mode, float *sink, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DECODE_H */
