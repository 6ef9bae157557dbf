/*
 * dn.h -- C ABI of libdn.so, the GB300 (sm_103a) DeltaNet recurrent-state path.
 *
 * Four operations make up the path a hybrid DeltaNet model runs for every
 * speculative verify step and every prompt:
 *
 *   dn_verify_block        run the draft block through the recurrence, keep one
 *                          state checkpoint per position
 *   dn_accept_greedy       argmax of each position's logits, longest matching
 *                          draft prefix
 *   dn_commit              make the checkpoint at the accepted position the
 *                          request's state (or keep the state when nothing was
 *                          accepted)
 *   dn_prefill_checkpoint  run a prompt through the recurrence and checkpoint the
 *                          state every `chunk` tokens for prefix caching
 *
 * The recurrence is the gated delta rule (Yang, Kautz, Hatamizadeh 2024,
 * "Gated Delta Networks"), the DeltaNet layer the pages serve:
 *
 *     S_t = g_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t
 *
 * S is a dv x dk matrix per (state set, head). A "state set" is one request's
 * state in one layer; callers may fold several layers of one request (or
 * several requests) into the leading dimension N of one call.
 *
 * LAYOUT. Every array is dense row-major (last index fastest), in device
 * memory, with the shapes given per function. The state is stored as the math
 * S itself: element (i, j) of a [dv][dk] tile, i over dv, j over dk.
 *
 * DTYPES. Two combinations are supported: io_dt = state_dt = DN_F16 (fp16
 * q/k/v/out and fp16 state, the 16-bit DeltaNet state of the pages) and
 * io_dt = state_dt = DN_F32. beta and g are always fp32. Inside a call the
 * state is carried in fp32; it is rounded (round-to-nearest-even) to the state
 * dtype only where it is stored.
 *
 * OWNERSHIP. The GPU entry points allocate nothing, keep no state between calls
 * and hold no pointer after a call returns (the prefix index below is a host-side
 * object the caller creates and destroys). All buffers belong to the caller.
 * Every call only enqueues work on `stream` (NULL means the legacy default
 * stream) and returns without synchronising; results are ready when the
 * stream reaches that point. Calls are deterministic: the same inputs give
 * bit-identical outputs.
 *
 * ERRORS. Every argument is checked on the host before anything is enqueued.
 * A malformed argument (null pointer where one is required, pointer not aligned
 * as stated, count out of range) returns DN_ERR_INVALID_ARG; a well-formed but
 * unsupported shape or dtype (dk or dv not 64/128, another dtype pair, another
 * chunk size) returns DN_ERR_UNSUPPORTED. In both cases nothing is enqueued.
 * DN_ERR_CUDA means a CUDA launch failed; the CUDA error has been consumed
 * with cudaGetLastError. Calls with a zero-sized leading count (N = 0, B = 0)
 * return DN_OK without enqueuing anything.
 *
 * Sources, cited by page title and section:
 *   [P1] "HyperQwen: 1,000 tok/s on a Single RTX 3090 Through Aggressive
 *        Recurrent-State Speculation", Technical Insight.
 *   [P2] "HyperQwen" (project README), The numbers behind that.
 *   [P3] "Qwen3.8-27B on a Single RTX 3090: How Calibrated Quantization and
 *        Speculative Decoding Hit 1,000 tok/s", Technical Insight.
 *   [P4] "HyperQwen on one RTX 3090: a first-time developer's guide to the
 *        381-token claim", What actually became faster?.
 */
#ifndef DN_H
#define DN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *dn_stream_t;

typedef enum {
    DN_OK = 0,
    DN_ERR_INVALID_ARG = 1,
    DN_ERR_UNSUPPORTED = 2,
    DN_ERR_CUDA = 3
} dn_status;

typedef enum { DN_F16 = 0, DN_F32 = 1 } dn_dtype;

/* Largest verify block (7 model drafts + 8 context drafts + 1 [P4]). */
#define DN_MAX_BLOCK 16
/* The only supported prefill checkpoint interval. */
#define DN_PREFILL_CHUNK 64

/*
 * dn_verify_block -- one verify block of T tokens, per-position checkpoints.
 *
 * The recurrent state of a DeltaNet layer grows with the verify width because
 * each verified position keeps its own state copy, so that any accepted prefix
 * can be committed ([P1]: 1.66 GiB at 15 drafts vs 0.88 GiB at 7; [P2]: a
 * speculating request holds its own pages of recurrent state). The block is at most
 * 16 tokens wide ([P4]).
 *
 * For every state set n < N and head h < H, starting from S = state_in[n][h]:
 *   for t = 0 .. T-1:  S = g[n][t][h] * S (I - beta[n][t][h] k k^T) + beta[n][t][h] v k^T
 *                      out[n][t][h][:] = S q          (with k, v, q of [n][t][h])
 *                      ckpt[n][t][h]   = S            (rounded to state_dt)
 *
 *   N        number of state sets (>= 0); layers of one request may be folded in
 *   H        heads per state set (>= 1)
 *   T        block width, 1 .. DN_MAX_BLOCK
 *   dk, dv   key / value head dims, each 64 or 128
 *   q, k     [N][T][H][dk]  io_dt            16-byte aligned, read only
 *   v        [N][T][H][dv]  io_dt            16-byte aligned, read only
 *   beta, g  [N][T][H]      fp32             4-byte aligned, read only
 *   state_in [N][H][dv][dk] state_dt         16-byte aligned, read only
 *   out      [N][T][H][dv]  io_dt            16-byte aligned, written
 *   ckpt     [N][T][H][dv][dk] state_dt      16-byte aligned, written
 * Output buffers must not overlap any input.
 */
dn_status dn_verify_block(int N, int H, int T, int dk, int dv,
                          dn_dtype io_dt, dn_dtype state_dt,
                          const void *q, const void *k, const void *v,
                          const float *beta, const float *g,
                          const void *state_in, void *out, void *ckpt,
                          dn_stream_t stream);

/*
 * dn_verify_block_deltas / dn_commit_deltas -- the verify block without per-position
 * checkpoints ("recompute on commit").
 *
 * A speculating request reserves a state copy per verified position ([P1]: 1.66 GiB
 * at 15 drafts vs 0.88 GiB at 7; [P2]: speculation holds state pages per request). This pair
 * keeps none: verify writes, per position, only the write strength of the delta rule
 *
 *   delta_t = beta_t (v_t - g_t S_{t-1} k_t)        (one fp32 per state row)
 *
 * so that S_t = g_t S_{t-1} + delta_t k_t^T; commit then rebuilds the accepted state
 * in place from the old state, delta_0..delta_{a-1}, k and g, in closed form:
 *
 *   S_a = (g_0 ... g_{a-1}) S_0 + sum_{s<a} (g_{s+1} ... g_{a-1}) delta_s k_s^T
 *
 * (one small tensor-core product per 64 state rows, with fp32-level accuracy). out is
 * identical to dn_verify_block's. The committed state agrees with dn_verify_block +
 * dn_commit on the same inputs to within one fp16 unit in the last place, and is equal
 * for nearly every element: both sum in fp32, in different orders.
 *
 * dn_verify_block_deltas: arguments as dn_verify_block, with
 *   delta    [N][T][H][dv] fp32, 16-byte aligned, written (instead of ckpt)
 * dn_commit_deltas: N, B, H, T, dk, dv, state_dt and accepted_len as dn_commit, with
 *   k        [N][T][H][dk] the block's keys (io dtype), 16-byte aligned
 *   g        [N][T][H] fp32 the block's gates
 *   delta    [N][T][H][dv] fp32 from dn_verify_block_deltas, 16-byte aligned
 *   state    [N][H][dv][dk], updated in place (must be dn_verify_block_deltas' state_in)
 * Both support the fp16 state / fp16 io pair only (DN_ERR_UNSUPPORTED otherwise).
 */
dn_status dn_verify_block_deltas(int N, int H, int T, int dk, int dv,
                                 dn_dtype io_dt, dn_dtype state_dt,
                                 const void *q, const void *k, const void *v,
                                 const float *beta, const float *g,
                                 const void *state_in, void *out, float *delta,
                                 dn_stream_t stream);
dn_status dn_commit_deltas(int N, int B, int H, int T, int dk, int dv, dn_dtype state_dt,
                           const void *k, const float *g, const float *delta,
                           const int32_t *accepted_len, void *state, dn_stream_t stream);

/*
 * dn_accept_workspace_bytes -- device workspace dn_accept_greedy needs.
 * Returns 0 for B < 1, T < 1 or V < 1.
 */
size_t dn_accept_workspace_bytes(int B, int T, int V);

/*
 * dn_accept_greedy -- greedy verification of B draft blocks.
 *
 * The verifier's logits are compared with the drafts and the accepted prefix
 * is kept ([P3], the verify step of the split-KV attention; "roughly 15 of
 * those 16 tokens were accepted per step" on document reproduction, [P4]):
 *
 *   target_ids[b][t]  = the lowest index v holding the maximum of logits[b][t][:]
 *                       (values compared as numbers, so -0.0 ties +0.0)
 *   accepted_len[b]   = the first t with draft_ids[b][t] != target_ids[b][t], or T
 *
 *   logits        [B][T][V] logit_dt (DN_F16 or DN_F32), 16-byte aligned;
 *                 any value but NaN (not checked): -inf marks a masked vocabulary
 *                 entry, and a row that is -inf throughout gives target 0 in
 *                 both dtypes
 *   draft_ids     [B][T] int32, 4-byte aligned
 *   target_ids    [B][T] int32, written
 *   accepted_len  [B] int32, written; stays on the device (dn_commit reads it
 *                 there, no host round trip is needed)
 *   workspace     >= dn_accept_workspace_bytes(B, T, V) bytes, 16-byte aligned.
 *                 It must hold zeros before its first use (cudaMemset once
 *                 after allocating it); every call leaves it ready for the
 *                 next one. Calls that may run concurrently need separate
 *                 workspaces.
 *   B >= 0, T >= 1, V >= 1; B * T * ceil(V / 8192) <= 2^31 - 1 (one CTA per
 *   row and 8,192-entry chunk), else DN_ERR_INVALID_ARG.
 */
dn_status dn_accept_greedy(int B, int T, int V, dn_dtype logit_dt, const void *logits,
                           const int32_t *draft_ids, int32_t *target_ids,
                           int32_t *accepted_len, void *workspace, size_t workspace_bytes,
                           dn_stream_t stream);

/*
 * dn_commit -- commit or roll back each state set to its accepted position.
 *
 * After verification the accepted prefix is kept and the rejected drafts are
 * discarded ([P3], verify step); for the recurrent state that means:
 *
 *   for n < N with a = accepted_len[n % B]:
 *     a == 0        : state[n] unchanged
 *     1 <= a <= T   : state[n] = ckpt[n][a-1]     (all H heads)
 *     otherwise     : state[n] unchanged (an out-of-range length is ignored)
 *
 *   N multiple of B, N * ceil(H * dv * dk * size / 32 KiB) <= 2^31 - 1 (one CTA
 *   per 32 KiB piece of a set); state set n belongs to request n % B (sets
 *   laid out [layer][request], n = layer * B + request).
 *   ckpt          [N][T][H][dv][dk] state_dt, 16-byte aligned (dn_verify_block's)
 *   accepted_len  [B] int32 in device memory, 4-byte aligned
 *   state         [N][H][dv][dk] state_dt, 16-byte aligned, updated in place
 */
dn_status dn_commit(int N, int B, int H, int T, int dk, int dv, dn_dtype state_dt,
                    const void *ckpt, const int32_t *accepted_len, void *state,
                    dn_stream_t stream);

/*
 * dn_prefill_checkpoint -- run P prompt tokens, checkpoint every `chunk` tokens.
 *
 * Prefix caching keeps the DeltaNet state next to the attention context so that
 * a later turn restores it instead of recomputing the prompt ([P1]; a second
 * question on a ~25,000-token document, 22.4 s -> 0.56 s to first token, [P4]).
 *
 * For every sequence n < N and head h < H, starting from S = state_in[n][h]
 * (zeros when state_in is NULL):
 *   for p = 0 .. P-1:  S = g S (I - beta k k^T) + beta v k^T;  out[n][p][h] = S q
 *                      if (p + 1) % chunk == 0:  S = round(S);  ckpt[n][(p+1)/chunk - 1][h] = S
 *   state_out[n][h] = round(S)
 * where round() rounds to state_dt. The carry at every chunk end is exactly the
 * stored checkpoint, so a run restored from ckpt[c] continues bit-identically to
 * the full run. The tail after the last full chunk writes no checkpoint.
 *
 *   N >= 0 sequences of equal length P >= 0; H >= 1; chunk == DN_PREFILL_CHUNK
 *   q, k      [N][P][H][dk] io_dt      v, out [N][P][H][dv] io_dt
 *   beta, g   [N][P][H] fp32
 *   state_in  [N][H][dv][dk] state_dt or NULL (zero initial state)
 *   ckpt      [N][P / chunk][H][dv][dk] state_dt; may be NULL when P < chunk
 *   state_out [N][H][dv][dk] state_dt; may be the same buffer as state_in
 * Alignment as for dn_verify_block. Other outputs must not overlap any input.
 */
dn_status dn_prefill_checkpoint(int N, int H, int P, int chunk, int dk, int dv,
                                dn_dtype io_dt, dn_dtype state_dt,
                                const void *q, const void *k, const void *v,
                                const float *beta, const float *g,
                                const void *state_in, void *out, void *ckpt,
                                void *state_out, dn_stream_t stream);

/*
 * dn_prefill_checkpoint_tc -- dn_prefill_checkpoint on the fifth-generation tensor cores.
 *
 * Same operation, arguments, layouts, ownership and errors as dn_prefill_checkpoint, for
 * fp16 io and state with dk = dv = 128 only (DN_ERR_UNSUPPORTED otherwise). The chunk is
 * computed in its 64-token form: grams, the WY factors U and W and the per-chunk state
 * products are tcgen05 MMAs with accumulators in tensor memory; the 64 x 64 triangular
 * inverse is solved in 16 x 16 blocks. Results agree with the oracle within the fp16
 * tolerance and restores from its checkpoints are bit-identical, but the rounding order
 * differs from dn_prefill_checkpoint, so the two engines' outputs are not bit-identical
 * to each other. On GB300 it is slower than dn_prefill_checkpoint on the 25,000-token
 * workload (the per-chunk chain of dependent steps, not the tensor pipe, bounds it).
 */
dn_status dn_prefill_checkpoint_tc(int N, int H, int P, int chunk, int dk, int dv, dn_dtype io_dt,
                                   dn_dtype state_dt, const void *q, const void *k, const void *v,
                                   const float *beta, const float *g, const void *state_in, void *out,
                                   void *ckpt, void *state_out, dn_stream_t stream);

/*
 * dn_accept_greedy_noalloc -- dn_accept_greedy without a caller-supplied workspace.
 *
 * The pages have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory at the point where they verify: a serving engine
 * that has handed almost all of the GPU's memory to its own page pool at start-up
 * and refuses further allocations, or plain C code embedded in such a host that
 * has no access to the host's allocator. Those callers pass the same inputs and
 * outputs as for dn_accept_greedy, and get the same results, but no workspace.
 *
 * The scratch lives in one fixed device array of DN_ACCEPT_NOALLOC_SCRATCH_BYTES
 * bytes inside libdn.so. Every GPU that loads the library holds that array until
 * the process exits. The call allocates nothing and frees nothing.
 *
 *   - Sizes: calls whose dn_accept_workspace_bytes(B, T, V) exceeds
 *     DN_ACCEPT_NOALLOC_SCRATCH_BYTES return DN_ERR_INVALID_ARG with nothing
 *     enqueued (about 1,600 verified positions at V = 151,936). Other arguments are
 *     checked as for dn_accept_greedy.
 *   - First call on a device: it looks up the array's device address once per
 *     CUDA context (with that device current; in the runtime's usual use, one
 *     primary context per device) and returns DN_ERR_CUDA if the lookup fails.
 *     Make that first call before any stream capture on that device. The address
 *     is cached under the context's unique id, so after cudaDeviceReset (which
 *     destroys the context and unloads the array) or in a second context on the
 *     same device the next call looks it up again instead of using a stale one.
 *   - Sharing: all calls on a device share the one array. The call clears the
 *     counters it needs on `stream` before its kernel runs, so leftovers of an
 *     earlier call do no harm; but two calls whose work overlaps on the GPU (on
 *     different streams, or from different threads) race on the array and give
 *     wrong results. Serialise them.
 */
#define DN_ACCEPT_NOALLOC_SCRATCH_BYTES (256u * 1024u)
dn_status dn_accept_greedy_noalloc(int B, int T, int V, dn_dtype logit_dt, const void *logits,
                                   const int32_t *draft_ids, int32_t *target_ids,
                                   int32_t *accepted_len, dn_stream_t stream);

/*
 * dn_context_drafts -- draft tokens copied from each request's own context.
 *
 * Single-user serving fills the later positions of the verify block (after the drafter's
 * 7) by copying from the request's context, since models often quote their input verbatim
 * ([P1]; [P4]: on document reproduction about 15 of 16 block tokens are accepted). The
 * pages do not say how the place to copy from is found; the rule here: the pattern is the
 * last n tokens of the context; take its latest earlier occurrence that has at least one
 * token after it, for the largest n in n_min..n_max that has one; the drafts are the up to
 * K tokens that follow it. No occurrence for any n: no drafts.
 *
 *   N          requests, >= 0
 *   stride     row pitch of context in tokens, 0 .. 2^27 - 1
 *   n_max      1 .. DN_MAX_NGRAM;  n_min  1 .. n_max
 *   K          drafts wanted, 1 .. DN_MAX_BLOCK
 *   context    [N][stride] int32 token ids (device); row r is prompt then generated tokens
 *   lengths    [N] int32 (device): row r uses context[r][0 .. lengths[r]); a length
 *              below 0 counts as 0 and one above stride as stride
 *   drafts     [N][K] int32 (device, written): the drafts, then -1 up to K
 *   count      [N] int32 (device, written): drafts found, 0 .. K
 *   match_len  [N] int32 (device, written) or NULL: the n used, 0 if none
 *
 * Reads L * 4 bytes per request; lengths are read on the device, so a caller that appends
 * accepted tokens on the device needs no host round trip. All pointers 4-byte aligned.
 * Returns DN_ERR_INVALID_ARG for bad sizes or pointers, DN_ERR_CUDA if the launch fails.
 */
#define DN_MAX_NGRAM 16
dn_status dn_context_drafts(int N, int stride, int n_max, int n_min, int K, const int32_t *context,
                            const int32_t *lengths, int32_t *drafts, int32_t *count,
                            int32_t *match_len, dn_stream_t stream);

/*
 * Prefix index for recurrent-state checkpoints (host memory, no GPU work).
 *
 * Prefix caching keeps the DeltaNet state so that a later turn restores it instead of
 * recomputing the prompt, and conversations with identical opening turns share state
 * across requests ([P1]; 22.4 s -> 0.56 s to first token on a ~25,000-token document,
 * [P4]). dn_prefill_checkpoint writes the state after every `chunk` tokens into
 * buffers the caller owns; this index maps token content to the caller's slot for
 * each such checkpoint. To serve a prompt, look up its longest cached prefix, pass
 * that checkpoint as state_in and prefill only the remaining tokens.
 *
 * Keys are exact: chunks are found by a 64-bit hash and then compared token by token,
 * so a collision never returns another prompt's state. Entries are evicted least
 * recently used (a lookup hit counts as a use). The index allocates host memory only;
 * calls are serialised by an internal lock.
 *
 * dn_prefix_cache_create  chunk >= 1 (use DN_PREFILL_CHUNK), capacity = max slots held;
 *                         NULL on bad arguments or out of memory.
 * dn_prefix_cache_insert  the state after tokens[0 .. position) is in `slot` (>= 0);
 *                         position a positive multiple of chunk. *evicted_slot receives
 *                         a slot the index dropped to make room (or replaced for this
 *                         prefix), -1 if none; the caller may reuse that slot's buffer.
 * dn_prefix_cache_lookup  longest cached prefix of tokens[0 .. n): *position (a multiple
 *                         of chunk, 0 if none) and *slot (-1 if none).
 * dn_prefix_cache_size    number of slots held.
 */
typedef struct dn_prefix_cache dn_prefix_cache;
dn_prefix_cache *dn_prefix_cache_create(int chunk, int capacity);
void dn_prefix_cache_destroy(dn_prefix_cache *c);
dn_status dn_prefix_cache_insert(dn_prefix_cache *c, const int32_t *tokens, int position,
                                 int32_t slot, int32_t *evicted_slot);
dn_status dn_prefix_cache_lookup(dn_prefix_cache *c, const int32_t *tokens, int n,
                                 int *position, int32_t *slot);
int dn_prefix_cache_size(dn_prefix_cache *c);

/*
 * dn_prefill_wait_timeouts -- diagnostics of the fp16 prefill kernels.
 *
 * The fp16 prefill kernels stream their inputs with the GPU's tensor-copy engine and
 * hand work between warp roles on shared-memory barriers. Every such wait is bounded
 * in time: it gives up after 1 second (1,000,000 us; a wait lasts a few microseconds
 * when the work it waits for progresses). When one runs out, the CTA counts the failure
 * here once, stops issuing copies and global stores, waits at most the same budget for
 * the copies and tensor-core operations it has already issued, and exits; the results
 * of that call are then invalid, and nothing hangs. Returns how many CTAs gave up since
 * the library was loaded on the current device (0 in correct operation), or 0xffffffff
 * if the counter could not be read. Synchronises the current device.
 */
unsigned int dn_prefill_wait_timeouts(void);

/*
 * dn_wait_selftest -- checks on the device the bounded waits of the prefill kernels.
 *
 * Launches one small kernel on `stream` that uses the kernels' own wait functions with a
 * time budget of `budget_us` microseconds:
 *   result[0] = 1: a wait on a shared-memory barrier nothing arrives on gave up after the
 *                  budget and raised the CTA's abort flag;
 *   result[1] = 1: after the one expected arrival, the same wait returned;
 *   result[2] = 1: the drain path: a 16-byte bulk copy from result[0..3] into shared memory
 *                  was in flight when a second wait ran out; the drain waited for it and
 *                  the copy landed with the bytes result[0..3] held at the launch;
 *   result[3] = 2: each of the two failures was counted once.
 * result: 4 int32 in device memory, 16-byte aligned, owned by the caller; its first 16
 * bytes are also the copy's source. 1 <= budget_us <= 1,000,000; the kernel takes about
 * two budgets. Errors: DN_ERR_INVALID_ARG (nothing launched), DN_ERR_CUDA (launch failed).
 */
dn_status dn_wait_selftest(int budget_us, int32_t *result, dn_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char *dn_status_string(dn_status s);

#ifdef __cplusplus
}
#endif

#endif /* DN_H */
