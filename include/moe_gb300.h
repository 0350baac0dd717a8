/*
 * moe_gb300.h -- C ABI of the routed mixture-of-experts layer served from a
 * GPU expert-slot cache (single GB300 GPU, sm_103a).
 *
 * The calls follow the problem statement in "Running DeepSeek-V4-Flash across
 * four free GPUs", section "What the expert cache actually does": the router
 * picks top_k experts per token, ensure_experts remaps the expert ids in place
 * onto cache slots, copy_missing moves only the misses from pinned host RAM,
 * and a grouped expert GEMM runs over the slot views.  The per-layer single
 * host synchronisation to read the router's picks is from "An elephant
 * through a straw", section "43 graphs, 43 syncs"; the (a,b) precision ladder
 * from its section "Not all six experts matter equally".
 *
 * Conventions for every call:
 *  - The caller owns every buffer it passes (device tensors, the pinned host
 *    bank, host miss lists).  The library owns only the opaque cache handle
 *    and the cache's device LRU arrays.
 *  - Pointers marked "device" must be device (or managed) memory; "host"
 *    pointers must be host memory.  Sizes are element counts unless stated.
 *  - Every call returns a moe_status.  Calls taking a cudaStream_t are
 *    asynchronous on that stream unless stated otherwise.  No call aborts,
 *    prints or synchronises the device implicitly.  moe_last_error() gives a
 *    message for the calling thread's last failure.
 *  - Errors that can only be seen on the device (an expert id >= E inside
 *    ids, a capacity overflow found while scanning) are reported through the
 *    device output words documented per call, never by a fault.
 *  - Matrices are row-major.  An MXFP4 expert is stored in the canonical
 *    layout: for gate w1 [I,H], up w3 [I,H], down w2 [H,I] in that order,
 *    codes [N][K/2] (two E2M1 codes per byte, element 2j in the low nibble)
 *    then E8M0 scales [N][K/32].  The 2-bit copy: codes [N][K/4] (element 4j+q
 *    at bits 2q..2q+1, value (q - 1.5) * scale) then E4M3 scales [N][K/32].
 *    The shared expert: E4M3 codes [N][K] then fp32 row scales [N].
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,   /* bad argument (null pointer, size, range, alignment) */
  MOE_ERR_CAPACITY = 2,  /* a single token needs more experts than the pool has slots */
  MOE_ERR_CUDA = 3,      /* a CUDA runtime call failed (message has the CUDA error) */
  MOE_ERR_TIMEOUT = 4,   /* a kernel's bounded wait gave up (grouped-GEMM mbarrier waits stop
                            after 1 s); reported through the call's d_error, the call itself
                            having returned MOE_OK when it was enqueued */
  MOE_ERR_NOMEM = 5      /* library-owned allocation failed */
} moe_status;

enum { MOE_FETCH = 0, MOE_LOOKUP = 1, MOE_FETCH_MARK_REST = 2 };
enum { MOE_TAG_FP4 = 0, MOE_TAG_INT2 = 1, MOE_TAG_DROP = 2 };
enum { MOE_POOL_FP4 = 0, MOE_POOL_INT2 = 1, MOE_POOL_SHARED = 2 };
enum { MOE_W1 = 0, MOE_W3 = 1, MOE_W2 = 2 };

/* Message of the calling thread's last failed call ("" if none).  The pointer
 * stays valid until the thread's next library call. */
const char* moe_last_error(void);
int moe_version(void);

/* Byte size of one expert in each format (0 if H or I is not a multiple of 32). */
size_t moe_fp4_expert_bytes(int H, int I);
size_t moe_int2_expert_bytes(int H, int I);
size_t moe_fp8_expert_bytes(int H, int I);

/* ---------------------------------------------------------------------------
 * Router: softmax over E logits, keep the top k, renormalise.
 * ("Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
 * cache actually does"; "An elephant through a straw", section "Not all six
 * experts matter equally".)
 *   logits   device fp32 [T, E], finite (non-finite logits give unspecified ids)
 *   topk_ids device int32 [T, k] out: the k largest logits of each row, in
 *            descending order, ties to the lower expert id
 *   topk_w   device fp32 [T, k] out: renorm != 0 -> exp(l_j - max) / sum over
 *            the kept of exp(l_i - max) (sums to 1); renorm == 0 -> the full
 *            softmax probability of each kept expert
 *   1 <= k <= min(E, 32), 1 <= E <= 2048, T >= 0 (T == 0 launches nothing).
 * ------------------------------------------------------------------------- */
moe_status moe_router_topk(const float* logits, int T, int E, int k, int renorm,
                           int32_t* topk_ids, float* topk_w, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Expert-slot cache ("What the expert cache actually does": a fixed number of
 * VRAM slots shared by all layers, LRU eviction, only misses copied from a
 * pinned host bank).  Key of an expert = layer * num_experts + expert.
 *   num_slots      S >= 1 slots of expert_bytes each at d_slots (device,
 *                  caller-owned, S * expert_bytes bytes, 16-byte aligned)
 *   h_bank         host memory holding num_layers * num_experts experts back to
 *                  back (key * expert_bytes); must be page-locked (registered
 *                  or cudaHostAlloc'ed); may be NULL for a cache that is only
 *                  ever filled by the caller (then moe_copy_missing fails)
 *   out            receives the handle; the cache starts empty.
 * Allocates the device LRU state (slot_key int32 [S], slot_stamp uint64 [S],
 * key_to_slot int32 [L*E], clock uint64) on the current device, synchronously.
 * ------------------------------------------------------------------------- */
typedef struct moe_cache moe_cache;

moe_status moe_cache_create(int num_slots, int num_layers, int num_experts,
                            size_t expert_bytes, void* d_slots, const void* h_bank,
                            moe_cache** out);
moe_status moe_cache_destroy(moe_cache* cache);
/* Empty every slot and reset the clock (asynchronous on stream). */
moe_status moe_cache_reset(moe_cache* cache, cudaStream_t stream);
/* Device pointers of the LRU state, for inspection (not to be freed). */
moe_status moe_cache_state(moe_cache* cache, int32_t** slot_key, uint64_t** slot_stamp,
                           int32_t** key_to_slot, uint64_t** clock);
/* Copy the LRU state to host arrays (slot_key [S], slot_stamp [S], clock [1]);
 * synchronous.  moe_cache_import restores it (key_to_slot is rebuilt) and
 * rejects states with out-of-range or duplicate keys. */
moe_status moe_cache_export(moe_cache* cache, int32_t* h_slot_key, uint64_t* h_slot_stamp,
                            uint64_t* h_clock);
moe_status moe_cache_import(moe_cache* cache, const int32_t* h_slot_key,
                            const uint64_t* h_slot_stamp, uint64_t clock);

/* ---------------------------------------------------------------------------
 * ensure_experts: remap expert ids of tokens [token_begin, T) and ranks
 * [rank_lo, rank_hi) onto slots, in first-appearance order (token-major,
 * then rank).  Entries holding a negative id are skipped.  ("Running
 * DeepSeek-V4-Flash across four free GPUs", section "What the expert cache
 * actually does": ids remapped in place onto cache slots before the expert
 * GEMM; its section "Step 7: Errors you will actually hit" for a cache too
 * small for one batch's experts, read here as the token-prefix chunking.)
 *   ids        device int32 [T, k] expert ids (< num_experts)
 *   slots_out  device int32 [T, k]; may alias ids (in-place remap, as the
 *              pages' ensure_experts).  Only the processed entries are written.
 *   mode MOE_FETCH:  the longest token prefix from token_begin whose distinct
 *              experts fit the S slots is processed.  Hits keep their slot;
 *              misses take empty slots (ascending index) then the least
 *              recently used slots not needed by this call.  Every distinct
 *              key's recency stamp becomes clock + its first-appearance index.
 *              The misses are listed as (key, slot) pairs in first-appearance
 *              order; the bytes must then be copied (moe_copy_missing) before
 *              the slots are read.
 *   mode MOE_LOOKUP: every token from token_begin is processed; hits get their
 *              slot and a fresh stamp, misses get -1; nothing is evicted or listed.
 *   mode MOE_FETCH_MARK_REST: as MOE_FETCH, and the entries of tokens from
 *              tokens_done on (within the rank range, non-negative ids) are set
 *              to -1 in slots_out, so a forward enqueued for all T tokens skips
 *              them; slots_out must not alias ids in this mode.
 *   d_miss_key, d_miss_slot  device int32 [>= min(S, num_experts)] out
 *   d_miss_count   device int32 [1] out: number of misses; on a device-detected
 *              error it is negative: -MOE_ERR_CAPACITY (a single token needs
 *              more than S slots) or -MOE_ERR_INVALID (an id >= num_experts);
 *              the cache state is then unchanged.
 *   d_tokens_done  device int32 [1] out: one past the last processed token;
 *              a value < T asks the caller to copy, compute and call again
 *              with token_begin = tokens_done.
 * Limits: k <= 64; (T - token_begin) * (rank_hi - rank_lo) <= 65536;
 * num_experts <= 4096.  One thread block; stream-ordered with other calls on
 * the same cache (calls on one cache must not overlap on the GPU).
 * ------------------------------------------------------------------------- */
moe_status moe_slot_ensure(moe_cache* cache, int layer_id, const int32_t* ids, int32_t* slots_out,
                           int T, int k, int rank_lo, int rank_hi, int mode, int token_begin,
                           int32_t* d_miss_key, int32_t* d_miss_slot, int32_t* d_miss_count,
                           int32_t* d_tokens_done, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * copy_missing: for each listed miss, copy expert_bytes from
 * h_bank + key * expert_bytes to d_slots + slot * expert_bytes with one
 * cudaMemcpyAsync on copy_stream, in list order.  ("Running DeepSeek-V4-Flash
 * across four free GPUs", section "What the expert cache actually does": only
 * the misses cross from the pinned host bank; "An elephant through a straw",
 * section "43 graphs, 43 syncs": one host synchronisation per layer reads the
 * miss list.)  ready (may be NULL) is
 * waited on by copy_stream first; done (may be NULL) is recorded on
 * copy_stream after the last copy, for the compute stream to wait on.
 *   h_miss_key, h_miss_slot  host int32 [n_miss] (the lists read back after
 *                            the per-layer synchronisation)
 * On a failed copy, the slots of that miss and of every later one are marked
 * empty on the device (the earlier copies stand), and MOE_ERR_CUDA is returned.
 * ------------------------------------------------------------------------- */
moe_status moe_copy_missing(moe_cache* cache, const int32_t* h_miss_key,
                            const int32_t* h_miss_slot, int n_miss, cudaStream_t copy_stream,
                            cudaEvent_t ready, cudaEvent_t done);
/* ---------------------------------------------------------------------------
 * Eviction policy.  "An elephant through a straw", section "Rig, model &
 * methodology": the best configuration evicts by LFU with frequency decay,
 * seeded from a routing trace.  MOE_EVICT_LRU (the default) is the policy of
 * "Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
 * cache actually does".  Under MOE_EVICT_LFU every key has an integer count:
 * each moe_slot_ensure call adds 1 to the count of every distinct key it
 * handles (FETCH and LOOKUP, hits and misses), capped at 2^20 - 1; the epoch
 * of a call is (ensure calls returned so far) / decay_calls, and a count last
 * written in epoch e0 is worth count >> min(31, epoch - e0); misses take empty
 * slots by ascending index, then the untouched slots of lowest worth, ties by
 * the older stamp.  moe_ladder_classify needs LRU caches (MOE_ERR_INVALID).
 * ------------------------------------------------------------------------- */
enum { MOE_EVICT_LRU = 0, MOE_EVICT_LFU = 1 };

/* Sets the policy for calls enqueued from now on; decay_calls >= 1 (LFU). */
moe_status moe_cache_set_policy(moe_cache* cache, int policy, int decay_calls);

/* Seeds the LFU counts from a routing trace: h_counts host uint32 [L*E]
 * (key = layer * E + expert), capped at 2^20 - 1, written in the current
 * epoch.  Synchronous (waits for the device). */
moe_status moe_cache_seed_frequency(moe_cache* cache, const uint32_t* h_counts);

/* Copies the LFU state to the host: counts [L*E], their epochs [L*E] and the
 * number of ensure calls counted so far.  Synchronous.  moe_cache_reset
 * clears all three. */
moe_status moe_cache_export_frequency(moe_cache* cache, uint32_t* h_counts, uint32_t* h_epochs,
                                      uint64_t* h_calls);

/* ---------------------------------------------------------------------------
 * Staging ring for predicted experts.  "An elephant through a straw", section
 * "Guessing the router two layers ahead": predicted experts are copied into a
 * small round-robin region appended to the slot buffer, so a guess never
 * evicts a resident expert; a wrong guess is overwritten by a later
 * prediction; a right one is in GPU memory when the router asks for it.
 *
 * moe_cache_set_staging(cache, R): ring slots S .. S+R-1 of the caller's slot
 * buffer (which must then hold S + R experts); allocates and clears the ring
 * state (0 removes it).  Synchronous.
 *
 * moe_prefetch(cache, layer, d_experts[n], ...): device int32 expert ids of
 * `layer`, in order.  Negative ids, ids repeated in the call, keys resident in
 * the cache and keys already staged are skipped; every other key takes ring
 * position pos % R (pos advances), displacing the key staged there.  Writes
 * the copy list (key, ring slot) of the guesses that still hold their slot
 * at the end of the call (the last min(new keys, R)) and its length to the
 * device arrays d_list_* (room for min(n, R) entries), to be copied by
 * moe_copy_missing_device.  An id >= E
 * makes the call a no-op with *d_list_count = -MOE_ERR_INVALID.  The cache's
 * own state (slots, stamps, counts) is never changed.
 *
 * When moe_slot_ensure later lists a staged key as a miss, moe_copy_missing_
 * device fills the cache slot from the key's staging slot (a device copy)
 * instead of the host bank.  Order the copies on one stream (or with events)
 * so that a staging slot's prefetch copy has landed before it is read and is
 * not overwritten while it is read.  moe_copy_missing (host lists, copy
 * engine) always copies from the bank.  moe_cache_reset clears the ring.
 * ------------------------------------------------------------------------- */
moe_status moe_cache_set_staging(moe_cache* cache, int num_stage);
moe_status moe_prefetch(moe_cache* cache, int layer_id, const int32_t* d_experts, int n,
                        int32_t* d_list_key, int32_t* d_list_slot, int32_t* d_list_count,
                        cudaStream_t stream);
/* Copies the ring to the host: the key staged in each ring slot (-1 = none)
 * and the next ring position.  Synchronous. */
moe_status moe_cache_export_staging(moe_cache* cache, int32_t* h_stage_key, uint32_t* h_pos);

/* ---------------------------------------------------------------------------
 * copy_missing driven from the device: reads the miss list and count written
 * by moe_slot_ensure (device int32 arrays) and copies every miss with GPU
 * loads of the pinned bank over the host-device link, stream-ordered on
 * `stream` -- no host synchronisation between ensure and the forward.  The
 * bank must be mapped into the device address space (true for pinned memory
 * on systems with unified addressing) and 16-byte aligned, as must be the
 * slot pool; otherwise MOE_ERR_INVALID.  An entry with an out-of-range key or
 * slot is not copied and, when d_error (device int32, may be null) is given,
 * sets *d_error to MOE_ERR_INVALID if it holds 0 (the caller clears it; the
 * slot that entry named keeps stale bytes).  max_ctas bounds the grid
 * (0: four CTAs of 256 threads per SM); a small grid leaves the SMs to
 * kernels that run concurrently, such as moe_expert_forward_overlap.
 * ------------------------------------------------------------------------- */
moe_status moe_copy_missing_device(moe_cache* cache, const int32_t* d_miss_key,
                                   const int32_t* d_miss_slot, const int32_t* d_miss_count,
                                   int max_ctas, int32_t* d_error, cudaStream_t stream);

/* Reads one 16-byte word of every 4 KB page of the cache's mapped host bank
 * (all num_layers * num_experts experts), stream-ordered on `stream`.  The
 * first GPU read of a page of pinned host memory runs far below the link's
 * rate (measured: 25-100 GB/s for an expert's first copy against ~170 GB/s
 * for later ones), so a server primes the bank once at setup and every miss
 * copy then runs at the link rate.  The bank is not modified.
 * MOE_ERR_INVALID if the bank is not mapped or not 16-byte aligned. */
moe_status moe_cache_prime_bank(moe_cache* cache, cudaStream_t stream);

/* The same copy for one part of the list: with n = *d_miss_count, part p of
 * n_parts copies the entries [n * p / n_parts, n * (p + 1) / n_parts) (integer
 * division; a part may be empty).  Launching parts 0..n_parts-1 in order with
 * an event after each lets moe_expert_forward_overlap_parts compute each
 * part's pairs as soon as that part has landed.  1 <= n_parts <=
 * MOE_MAX_COPY_PARTS, else MOE_ERR_INVALID.  moe_copy_missing_device is part 0
 * of 1. */
#define MOE_MAX_COPY_PARTS 4
moe_status moe_copy_missing_device_part(moe_cache* cache, const int32_t* d_miss_key,
                                        const int32_t* d_miss_slot, const int32_t* d_miss_count,
                                        int part, int n_parts, int max_ctas, int32_t* d_error,
                                        cudaStream_t stream);

/* The same copy restricted to the bytes [byte_begin, byte_end) of every listed
 * expert (both multiples of 16, byte_end <= the expert size, else
 * MOE_ERR_INVALID).  With the FP4 layout, [0, 2 * (H*I/2 + H*I/32)) holds w1
 * and w3 (gate/up) and the rest w2 (down): copying the gate/up range first lets
 * moe_expert_forward_overlap_staged start the missed experts' gate/up work
 * while their down matrices are still crossing the link. */
moe_status moe_copy_missing_device_range(moe_cache* cache, const int32_t* d_miss_key,
                                         const int32_t* d_miss_slot, const int32_t* d_miss_count,
                                         size_t byte_begin, size_t byte_end, int max_ctas,
                                         int32_t* d_error, cudaStream_t stream);
/* Both at once: part `part` of n_parts of the list (as moe_copy_missing_device_
 * part divides it), bytes [byte_begin, byte_end) of each of its experts. */
moe_status moe_copy_missing_device_slice(moe_cache* cache, const int32_t* d_miss_key,
                                         const int32_t* d_miss_slot, const int32_t* d_miss_count, int part,
                                         int n_parts, size_t byte_begin, size_t byte_end, int max_ctas,
                                         int32_t* d_error, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Whole-layer streaming for prefill past the crossover.  "Running DeepSeek-
 * V4-Flash across four free GPUs", section "What the expert cache actually
 * does": above T * top_k >= num_experts prefill streams whole expert layers
 * instead of fetching slots, because a chunk touches most of the layer anyway;
 * section "Step 7" ("moe_cache_size=128 is too small"): with prefill overlap
 * two full expert-layer buffers are in use.  Copies all num_experts experts of
 * layer `layer_id` (bytes layer_id * E * B .. +E * B of the key-major pinned
 * bank) into the device buffer d_buf (E * B bytes) with one cudaMemcpyAsync
 * on `stream` (the copy engine: no SM time taken from the compute).  The
 * buffer then serves as an E-slot pool whose slot e holds expert e, for
 * moe_expert_prefill.  The slot cache is not involved.
 * ------------------------------------------------------------------------- */
moe_status moe_copy_layer(const void* h_bank, int layer_id, int num_experts, size_t expert_bytes,
                          void* d_buf, cudaStream_t stream);

/* Test hook: make the copy with list index `index` of later moe_copy_missing
 * calls fail on the host, as if cudaMemcpyAsync had returned an error
 * (index < 0 disarms).  Nothing is issued to the device for a failed copy. */
moe_status moe_debug_fail_copy(moe_cache* cache, int index);

/* ---------------------------------------------------------------------------
 * Precision ladder (a, b) over an FP4 cache and a 2-bit-copy cache
 * ("An elephant through a straw", section "Not all six experts matter
 * equally").  Ranks are 1-based on the page; here ranks [0, a) always use
 * FP4 (fetched if missing); ranks [a, b) use FP4 if resident, else the 2-bit
 * copy (fetched if missing); ranks [b, k) use FP4 if resident, else the 2-bit
 * copy if resident, else are dropped.  Passes run over the whole chunk in
 * that order; the chunk is the longest token prefix from token_begin whose
 * distinct rank-[0,a) experts fit the FP4 cache and whose distinct
 * rank-[a,b) experts fit the 2-bit cache.  Survivor weights are renormalised.
 *   ids, w      device int32 / fp32 [T, k] (router output)
 *   slots_out   device int32 [T, k]: slot in the tagged pool, -1 if dropped
 *   tags_out    device int8  [T, k]: MOE_TAG_FP4 / MOE_TAG_INT2 / MOE_TAG_DROP
 *   w_out       device fp32  [T, k]: renormalised weights, 0 if dropped
 *   miss lists and counts per pool as for moe_slot_ensure (counts negative on
 *   a device-detected error); d_tokens_done as for moe_slot_ensure.
 * Limits as moe_slot_ensure; 1 <= a <= b <= k.
 * ------------------------------------------------------------------------- */
moe_status moe_ladder_classify(moe_cache* fp4_cache, moe_cache* int2_cache, int layer_id,
                               const int32_t* ids, const float* w, int T, int k, int a, int b,
                               int token_begin, int32_t* slots_out, int8_t* tags_out,
                               float* w_out, int32_t* d_miss4_key, int32_t* d_miss4_slot,
                               int32_t* d_miss4_count, int32_t* d_miss2_key,
                               int32_t* d_miss2_slot, int32_t* d_miss2_count,
                               int32_t* d_tokens_done, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Grouping of (token, rank) pairs by expert (the permutation in front of a
 * grouped GEMM; "Running DeepSeek-V4-Flash across four free GPUs", section
 * "All four workers die, but only on prompts over 32 tokens").
 *   ids      device int32 [T, k]; negative ids are left out
 *   offsets  device int32 [E + 1] out: first position of each expert in perm
 *   perm     device int32 [T * k] out: flat pair indices t*k + j stably sorted
 *            by id (positions >= offsets[E] are left unwritten)
 *   d_error  device int32 [1] out: 0, or MOE_ERR_INVALID if an id >= E
 * ------------------------------------------------------------------------- */
moe_status moe_group_pairs(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                           int32_t* perm, int32_t* d_error, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped expert MLP + combine.  For every kept pair (t, j):
 * h = SiLU(W1 x_t) * (W3 x_t), o = W2 h, and
 * y_t = sum_j w[t,j] * o[t,j] + shared(x_t), rounded to bf16.
 * ("Running DeepSeek-V4-Flash across four free GPUs", sections "The model"
 * and "What the expert cache actually does": MXFP4 routed experts run as a
 * grouped GEMM over the cache slots; "An elephant through a straw", opening
 * section: MXFP4 experts of 13,369,344 bytes and the 2-bit copy.)
 * ------------------------------------------------------------------------- */
typedef struct {
  int H, I;                    /* hidden and intermediate sizes, multiples of 32 */
  const uint8_t* fp4_slots;    /* device: FP4 slot s at fp4_slots + s * moe_fp4_expert_bytes */
  int fp4_num_slots;
  const uint8_t* int2_slots;   /* device or NULL: 2-bit-copy slot s at int2_slots + s * bytes */
  int int2_num_slots;
  const uint8_t* shared;       /* device or NULL: the FP8 shared expert */
} moe_expert_views;

/* Workspace bytes moe_expert_forward needs for T tokens of k pairs each. */
size_t moe_expert_forward_workspace(const moe_expert_views* v, int T, int k);

/*   x        device bf16 [T, H] (uint16 bit patterns)
 *   slots    device int32 [T, k]: slot of each pair in the pool given by tags
 *   tags     device int8 [T, k] or NULL (all MOE_TAG_FP4); MOE_TAG_DROP pairs
 *            and pairs with a negative slot are skipped
 *   w        device fp32 [T, k] router weights
 *   y        device bf16 [T, H] out
 *   workspace device, >= moe_expert_forward_workspace bytes, 256-byte aligned
 *   d_error  device int32 [1] out: 0, or MOE_ERR_INVALID if a slot >= the
 *            pool's slot count (the pair is then skipped)
 * Numerics: weights are decoded exactly; activations are held in fp16 with a
 * per-token power-of-two scale.  On the warp-level tensor-core path (see
 * moe_set_option) products accumulate in fp32 (bf16 operands for a 128-weight
 * chunk whose E8M0 scales leave [2^-12, 2^13]); on the CUDA-core path
 * 32-weight partial sums accumulate in fp16 and are scaled and summed in fp32;
 * from 256 pairs above that path's token limit the tcgen05 grouped GEMM runs
 * (fp16 or bf16 operands, fp32 accumulate, h in bf16).  The combine runs in
 * fp32 in rank order.
 * Above 4096 pairs per call the grouped-GEMM path of moe_expert_prefill is
 * taken (FP4 pool only, tags must be NULL). */
moe_status moe_expert_forward(const moe_expert_views* v, const uint16_t* x, int T, int k,
                              const int32_t* slots, const int8_t* tags, const float* w,
                              uint16_t* y, void* workspace, size_t workspace_bytes,
                              int32_t* d_error, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * moe_expert_forward for a chunk whose missed experts are still being copied
 * in.  On the pages the copies of a layer's misses take most of its time
 * ("An elephant through a straw", section "43 graphs, 43 syncs"; "Running
 * DeepSeek-V4-Flash across four free GPUs", section "What the expert cache
 * actually does"); here the pairs routed to resident experts, and the shared
 * expert, are computed while the copies run, and only the pairs whose slot is
 * on the miss list wait for them.
 *   slots, w, x, y  as moe_expert_forward (FP4 pool, no tags)
 *   d_miss_slot     device int32: the chunk's miss list slots (as written by
 *                   moe_slot_ensure); d_miss_count device int32 [1]: its length
 *                   (negative counts as 0; at most max_miss entries are read)
 *   copies_done     event recorded after this chunk's copies (on any stream),
 *                   or NULL when they are already complete
 *   workspace       device, >= moe_expert_forward_overlap_workspace bytes,
 *                   256-byte aligned
 *   d_error         as moe_expert_forward (cleared by the call)
 * The result equals moe_expert_forward's for the same slots (one combine over
 * all pairs in rank order).  Limits: T * k <= 4096, FP4 pool, no tags.
 *
 * moe_expert_forward_overlap_parts splits the missed pairs further by the part
 * of the miss list (as moe_copy_missing_device_part divides it) their slot is
 * in: after the first pass the stream waits on parts_done[p] and computes
 * part p's pairs, for p = 0..n_parts-1, so only the last part's pairs follow
 * the last copy.  parts_done: host array of n_parts events (NULL entries:
 * already complete); 1 <= n_parts <= MOE_MAX_COPY_PARTS.  The workspace size
 * covers every n_parts; the result is the same as moe_expert_forward's.
 *
 * moe_expert_forward_overlap_staged: the missed experts arrive in stages,
 * their gate/up matrices (event gateup_ready) and then their down matrices in
 * n_down_parts parts of the miss list (events down_ready[0..n_down_parts-1],
 * as moe_copy_missing_device_slice divides the list); the missed pairs'
 * gate/up work waits only for the first event, the down work of the pairs of
 * part q for down_ready[q] (the CUDA-core path waits for the last).  NULL
 * events: already complete; 1 <= n_down_parts <= MOE_MAX_COPY_PARTS.  Same
 * workspace and result as moe_expert_forward_overlap.
 * ------------------------------------------------------------------------- */
size_t moe_expert_forward_overlap_workspace(const moe_expert_views* v, int T, int k);
moe_status moe_expert_forward_overlap(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                      const int32_t* slots, const float* w, const int32_t* d_miss_slot,
                                      const int32_t* d_miss_count, int max_miss, cudaEvent_t copies_done,
                                      uint16_t* y, void* workspace, size_t workspace_bytes,
                                      int32_t* d_error, cudaStream_t stream);
moe_status moe_expert_forward_overlap_staged(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                             const int32_t* slots, const float* w, const int32_t* d_miss_slot,
                                             const int32_t* d_miss_count, int max_miss, cudaEvent_t gateup_ready,
                                             int n_down_parts, const cudaEvent_t* down_ready, uint16_t* y,
                                             void* workspace, size_t workspace_bytes, int32_t* d_error,
                                             cudaStream_t stream);
moe_status moe_expert_forward_overlap_parts(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                            const int32_t* slots, const float* w, const int32_t* d_miss_slot,
                                            const int32_t* d_miss_count, int max_miss, int n_parts,
                                            const cudaEvent_t* parts_done, uint16_t* y, void* workspace,
                                            size_t workspace_bytes, int32_t* d_error, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped-GEMM expert MLP for prefill-sized batches ("Running DeepSeek-V4-
 * Flash across four free GPUs", section "All four workers die, but only on
 * prompts over 32 tokens": past T * top_k >= num_experts the experts run as
 * one grouped GEMM over all tokens routed to each).  Same inputs and result
 * as moe_expert_forward for an FP4 pool without tags or shared expert; the
 * pairs are grouped by slot (moe_group_pairs), each group's activations are
 * gathered, and gate/up (with SwiGLU) and down run as tcgen05 bf16 MMAs with
 * fp32 accumulators in tensor memory; weights are decoded to bf16 exactly,
 * h is rounded to bf16.  Requires H and I multiples of 512, the FP4 pool
 * only, d_error non-null.  d_error receives MOE_ERR_TIMEOUT if a pipeline
 * wait on the device gave up (the output is then unspecified).
 * ------------------------------------------------------------------------- */
size_t moe_expert_prefill_workspace(const moe_expert_views* v, int T, int k);
moe_status moe_expert_prefill(const moe_expert_views* v, const uint16_t* x, int T, int k,
                              const int32_t* slots, const float* w, uint16_t* y, void* workspace,
                              size_t workspace_bytes, int32_t* d_error, cudaStream_t stream);

/* moe_expert_prefill with a precision mode.  MOE_PREC_W4A16 (the pages'
 * semantics, = moe_expert_prefill): activations bf16.  MOE_PREC_A_MXFP4 (not on
 * the pages; the tensor cores' block-scaled FP4 format): x, per token along H,
 * and h, per routed pair along I, are quantised to MXFP4 by the OCP MX rule of
 * moe_mx_quantize before their products, which then run on the exact
 * quantised values (bf16 MMA, fp32 accumulate).  Same workspace; an unknown
 * mode gives MOE_ERR_INVALID. */
#define MOE_PREC_W4A16 0
#define MOE_PREC_A_MXFP4 1
moe_status moe_expert_prefill_prec(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                   const int32_t* slots, const float* w, int prec_mode, uint16_t* y,
                                   void* workspace, size_t workspace_bytes, int32_t* d_error,
                                   cudaStream_t stream);

/* OCP MX quantisation (OCP Microscaling Formats (MX) Specification v1.0) of a
 * bf16 matrix to MXFP4, the activation step of MOE_PREC_A_MXFP4:
 *   x       device bf16 [rows, K], row-major, 16-byte aligned; K % 32 == 0
 *   codes   device uint8 [rows, K/2] out, 16-byte aligned: element 2j in the
 *           low nibble of byte j (E2M1 codes)
 *   scales  device uint8 [rows, K/32] out: one E8M0 byte per 32-element block
 * Per block: X = 2^(floor(log2 amax) - 2) (byte clamped to [0, 254]; an
 * all-zero block takes 2^-127), element = E2M1 value nearest to v / X with
 * ties to the even code, saturated at 6, zero magnitudes as +0.  Stream-
 * ordered; MOE_ERR_INVALID on bad sizes, null or misaligned pointers. */
moe_status moe_mx_quantize(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                           cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * moe_expert_forward without a caller-provided workspace.  The pages have no
 * counterpart; this serves callers that cannot allocate device memory: hosts
 * that hand a module a stream but own the device-memory budget, and serving
 * loops that forbid cudaMalloc after start-up (it can synchronise the device
 * and fail once memory is committed).  The scratch is a fixed 32 MiB array in
 * the library's device memory (held by every GPU that loads the library until
 * the process exits), enough for T = 64 tokens of top-8 at H = 4096,
 * I = 2048; larger calls return MOE_ERR_INVALID.  The caller still passes the
 * inputs and outputs; arguments as moe_expert_forward (decode path only:
 * T * k <= 4096).  The first call on a device looks up the scratch's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The call allocates nothing.  All calls
 * share the one scratch, which keeps the last call's contents (nothing in it
 * needs to start at zero): calls that overlap on the GPU race, so issue them
 * on one stream or order them.  The looked-up address is kept for the life of
 * the process: after cudaDeviceReset (or any teardown of the device's primary
 * context) it no longer names the scratch, so do not call this entry point on
 * that device again in the same process.
 * ------------------------------------------------------------------------- */
moe_status moe_expert_forward_noalloc(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                      const int32_t* slots, const int8_t* tags, const float* w,
                                      uint16_t* y, int32_t* d_error, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Process-wide tuning options (not on the pages).  MOE_OPT_MMA_MAX_TOKENS:
 * decode calls of 2 up to this many tokens run their FP4 and shared-expert
 * pairs on the tensor cores in decode-sized groups (default 64; 0 = never);
 * larger ones take the tcgen05 grouped GEMM from 256 pairs, and the CUDA-core
 * GEMV below that (and at one token).  MOE_OPT_MX8_MIN_TOKENS: of those
 * calls, the ones with at least this many tokens use the block-scaled
 * tcgen05 GEMM (tcgen05.mma.kind::mxf8f6f4: E2M1 weights as stored, the
 * activations and h split into two E4M3 terms with a power-of-two scale per
 * 32 elements, which holds a bf16 value exactly but for subnormal low terms),
 * the others the warp-level kernels (mma.sync); 0 = never.  It needs at most
 * 64 tokens, H and I multiples of 512 up to 4096, fp4_slots 32-byte and x
 * 8-byte aligned, and falls back to the warp-level kernels otherwise.  The previous value goes to
 * *old_value (may be null).  MOE_ERR_INVALID for an unknown option or a
 * negative value.  Set them between calls, not while another thread issues
 * forward calls.
 * ------------------------------------------------------------------------- */
enum { MOE_OPT_MMA_MAX_TOKENS = 0, MOE_OPT_MX8_MIN_TOKENS = 1 };
moe_status moe_set_option(int option, int value, int* old_value);

/* Diagnostic (not on the pages): the block-scaled FP4 tensor rate of this GPU.
 * One CTA per SM issues `iters` groups of four tcgen05.mma.kind::mxf4 (M = 128,
 * N = 256, K = 64, E8M0 unit scales) from shared memory into one tensor-memory
 * accumulator, with no data movement; *tflops receives the dense TFLOP/s
 * (2 M N K per MMA) measured with CUDA events on `stream`.  The call
 * synchronises the stream (and allocates 4 bytes of device memory for its
 * status).  iters a positive multiple of 64, else MOE_ERR_INVALID;
 * MOE_ERR_TIMEOUT if the completion wait gave up. */
moe_status moe_fp4_mma_peak(int iters, double* tflops, cudaStream_t stream);

/* Decode one matrix of one slot to fp32 [N, K] (test hook; values are exact). */
moe_status moe_dequant_debug(const moe_expert_views* v, int pool, int slot, int matrix,
                             float* out, cudaStream_t stream);

/* Next layer's input for a stack of layers: x_next = bf16(y / sqrt(mean(y^2) + eps))
 * per token, computed in fp32 (a weightless RMSNorm).  y and x_next device bf16 [T, H]. */
moe_status moe_rms_carry(const uint16_t* y, int T, int H, float eps, uint16_t* x_next,
                         cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Per-kernel timing: when enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on its launching stream.
 * moe_profile_enable(1) clears the record and starts collecting; (0) stops.
 * moe_profile_query synchronises on the recorded events and returns, for one
 * kernel id, the summed elapsed milliseconds and the number of launches.
 * moe_profile_timeline synchronises likewise and writes, in recording order,
 * up to `max` records (host arrays of length >= max): the kernel id and the
 * start and stop times in milliseconds relative to the start of the first
 * record, whatever stream each was launched on; *n receives the number of
 * records held (which may exceed max).  MOE_ERR_INVALID on a null pointer or
 * max < 0.
 * ------------------------------------------------------------------------- */
enum {
  MOE_K_ROUTER = 0, MOE_K_ENSURE, MOE_K_LADDER, MOE_K_GROUP, MOE_K_PLAN, MOE_K_GATEUP,
  MOE_K_DOWN, MOE_K_COMBINE, MOE_K_CARRY, MOE_K_GEMM_GATEUP, MOE_K_GEMM_DOWN, MOE_K_COPY, MOE_K_COUNT
};
moe_status moe_profile_enable(int enable);
moe_status moe_profile_query(int kernel, double* total_ms, int* launches);
moe_status moe_profile_timeline(int max, int32_t* kernel, double* start_ms, double* stop_ms, int* n);

/* Test hook for failure detection without a fault: launches one thread that
 * waits on an mbarrier nothing arrives on, with the library's bounded wait and
 * a limit of limit_ns (at most 2 s); *d_status (device int32) becomes
 * MOE_ERR_TIMEOUT when the wait gives up.  The context stays usable. */
moe_status moe_debug_timeout_probe(int64_t limit_ns, int32_t* d_status, cudaStream_t stream);

/* Runs a tiny router + cache + copy round trip and a tiny expert forward
 * (H = 64, I = 32, two all-ones FP4 experts, x = 1: every output exactly 2^17)
 * on the current device and checks them (synchronous).  MOE_OK means the
 * library executes here. */
moe_status moe_selftest(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
