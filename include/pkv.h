/*
 * pkv.h -- C ABI of libpkv: GQA attention over a paged KV cache on GB300 (sm_103a).
 *
 * The library is the data-parallel hot path of a nano-vLLM-style inference
 * step, as the pages describe it:
 *
 *   a1  pkv_slot_mapping     where each new token's K/V row lives in the pool
 *   a2  pkv_store_kvcache    scatter the new K/V rows into the block pool
 *   a3  pkv_prefill_varlen   varlen prefill attention, position-offset causal mask
 *   a4  pkv_decode           single-token decode attention over the block tables
 *   a5  pkv_sample           temperature sampling by exponential race
 *   f2  pkv_rope_store_kvcache  rotary embedding of Q/K fused into the a2 write
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is DEVICE memory owned by the caller, unless stated.
 *   The library keeps no pointer after a call returns and frees nothing.
 * - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *   NULL is the legacy default stream).  No call synchronises with the host,
 *   reads device data on the host, or allocates device memory; scratch space
 *   comes from a caller-provided workspace whose size a *_workspace_size call
 *   reports.  `max_*` bounds are passed in for the same reason.
 * - Host-checkable errors (null pointers, unsupported shapes, bad sizes) return
 *   a non-zero pkv_status before anything is launched.  A failed launch
 *   returns PKV_ERR_CUDA.  Errors only the device can see (a block id outside
 *   the pool, a decreasing cu_seqlens, a temperature <= 0, a pipeline wait that
 *   ran out) are recorded in a per-device error word read by
 *   pkv_get_device_error(); the kernel then skips the offending access.
 * - K/V pools are laid out [num_blocks, block_size, num_kv_heads, head_dim] in
 *   bf16, one pool per layer for K and one for V.  Block tables are int32
 *   [num_seqs, max_blocks_per_seq], row s listing sequence s's physical block
 *   ids in logical order, padded with -1.  Supported: head_dim = 128,
 *   block_size a multiple of 256, and num_heads = G * num_kv_heads with a
 *   group size G of 1, 2, 4 or 8 (MHA, and GQA with 2, 4 or 8 query heads
 *   sharing each KV head -- Visual atlas fig. 18; Qwen3-0.6B has G = 2);
 *   query head h reads KV head h / G.  Anything else returns
 *   PKV_ERR_UNSUPPORTED.
 * - bf16 tensors are passed as pkv_bf16 (the raw 16-bit pattern).
 *
 * Citations name the page and the figure or section that defines the step.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;     /* raw bfloat16 bits */
typedef void *pkv_stream_t;    /* cudaStream_t */

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent sizes */
    PKV_ERR_UNSUPPORTED = 2,   /* shape or device outside the supported set */
    PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    PKV_ERR_CUDA = 4           /* a CUDA runtime/driver call failed */
} pkv_status;

/* Device-side error codes (first one recorded wins). */
enum {
    PKV_DEVERR_NONE = 0,
    PKV_DEVERR_BLOCK_ID = 1,     /* block table entry outside [0, num_blocks) */
    PKV_DEVERR_SLOT = 2,         /* slot_mapping entry >= num_blocks * block_size */
    PKV_DEVERR_SEQLENS = 3,      /* cu_seqlens decreasing, q_len > k_len, or a length above its max_* bound */
    PKV_DEVERR_TEMPERATURE = 4,  /* temperature <= 0, inf or NaN */
    PKV_DEVERR_TIMEOUT = 5,      /* an mbarrier wait exceeded its limit */
    PKV_DEVERR_BLOCK_TABLE = 6,  /* a position past max_blocks_per_seq * block_size */
    PKV_DEVERR_PLAN = 7          /* the prefill workspace holds no plan for these arguments */
};

/* ABI version; bumped on any signature change. */
PKV_API int32_t pkv_abi_version(void);

/* Human-readable name of a pkv_status.  Static storage; never NULL. */
PKV_API const char *pkv_status_string(pkv_status status);

/*
 * a1. Slot of every new token.
 * Visual atlas (diomchen.github.io/reference/visual-atlas.html), figure
 * "T=5, block_size=2, block_table=[3,0,4]": slot = block_table[pos / bs] * bs
 * + pos % bs.  The new tokens of sequence s are its last q_len positions:
 * positions k_len - q_len .. k_len - 1 (atlas fig. 26: after a prefix hit the
 * query is shorter than the keys; Nano-vLLM overview, Sequence counters: a
 * decode feeds the one token without KV).
 *
 *   cu_seqlens_q  int32 [num_seqs + 1]; NULL means one new token per sequence
 *                 (decode: token i belongs to sequence i, total_q == num_seqs)
 *   cu_seqlens_k  int32 [num_seqs + 1] running key offsets, or NULL
 *   context_lens  int32 [num_seqs] keys per sequence, or NULL; exactly one of
 *                 cu_seqlens_k / context_lens is non-NULL
 *   slot_mapping  int32 [total_q] output, packed token order.  A token whose
 *                 position falls outside its block table gets -1 and
 *                 PKV_DEVERR_BLOCK_TABLE / PKV_DEVERR_BLOCK_ID is recorded.
 */
PKV_API pkv_status pkv_slot_mapping(const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            const int32_t *context_lens, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, int32_t num_seqs, int32_t total_q,
                            int32_t block_size, int32_t num_blocks, int32_t *slot_mapping,
                            pkv_stream_t stream);

/*
 * a2. Scatter new K/V rows into the pools: k_cache[slot / bs, slot % bs] = k[i],
 * v_cache likewise, for i < n_tokens.  nano-vLLM offline explainer
 * (3479845.xyz/nano-vllm/nano-vllm-offline), accuracy & scope box: the input
 * tokens write their KV first; interactive guide (blog-mushroom.pages.dev)
 * ch. 08: the KV cache is written during attention.
 *
 *   k, v            bf16 [n_tokens, num_kv_heads, head_dim]; token i starts at
 *                   element i * k_token_stride (resp. v_token_stride), which
 *                   must be a multiple of 8 and >= num_kv_heads * head_dim
 *                   (so k/v may be views into a fused QKV buffer)
 *   slot_mapping    int32 [n_tokens]; slot < 0 skips the row (padding)
 *   k_cache/v_cache bf16 pools, written in place
 * A slot >= num_blocks * block_size is skipped and PKV_DEVERR_SLOT recorded.
 * Bit-exact copy.  Rows with equal slots race (last writer unspecified).
 */
PKV_API pkv_status pkv_store_kvcache(const pkv_bf16 *k, const pkv_bf16 *v, int64_t n_tokens,
                             int64_t k_token_stride, int64_t v_token_stride,
                             const int32_t *slot_mapping, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                             int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                             int32_t head_dim, pkv_stream_t stream);

/*
 * f2. Rotary position embedding fused into the KV write.
 * Visual atlas, fig. 19: each head of d elements forms d/2 two-dimensional
 * pairs; pair i of a token at position p turns by p * rope_base^(-2i/d)
 * radians, (a, b) -> (a cos - b sin, b cos + a sin).  Q and K are rotated,
 * V is not.  Pair i couples elements i and i + d/2 of the head.
 *
 * For each token t < n_tokens: every head of q[t] (num_heads x head_dim,
 * token stride q_token_stride elements) is rotated by positions[t] into
 * q_out[t]; every head of k[t] is rotated and written, with v[t] unchanged,
 * to pool slot slot_mapping[t] exactly as pkv_store_kvcache does (a negative
 * slot skips the K/V write but still rotates q; a slot >= num_blocks *
 * block_size is recorded as PKV_DEVERR_SLOT with info = t and skipped).
 * The angle is reduced modulo 2 pi exactly, in 64-bit fixed-point turns (error
 * below 1e-6 rad even at |position| = 2^31); sine and cosine come from the
 * hardware approximation (within 4e-7 absolute on [-pi, pi]), the rotation
 * runs in fp32, and each result is rounded once to bf16.
 *
 * q and q_out are both NULL (rotate and store K only) or both non-NULL;
 * q_out may equal q (in place, equal strides) but must not partly overlap it
 * or any other argument.  Supported: head_dim a multiple of 16 up to 256,
 * token strides multiples of 8 elements, 16-byte aligned pointers; otherwise
 * PKV_ERR_UNSUPPORTED.  rope_base must be positive and finite.
 */
PKV_API pkv_status pkv_rope_store_kvcache(const pkv_bf16 *q, int64_t q_token_stride, pkv_bf16 *q_out,
                                  int64_t q_out_token_stride, const pkv_bf16 *k, int64_t k_token_stride,
                                  const pkv_bf16 *v, int64_t v_token_stride, const int32_t *positions,
                                  int64_t n_tokens, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, double rope_base, const int32_t *slot_mapping,
                                  pkv_bf16 *k_cache, pkv_bf16 *v_cache, int32_t num_blocks,
                                  int32_t block_size, pkv_stream_t stream);

/*
 * a3. Varlen prefill attention over the paged cache.
 * Visual atlas, figure "cu_seqlens=[0,3,5]" (packed requests), figs. 16-17
 * (softmax(scale QK^T + mask) V; diagonal kept; a cached chunk keeps its
 * position offset), fig. 18 (query heads share K/V heads), fig. 22 (blockwise
 * evaluation without materialising scores).
 *
 * For sequence s with q_len = cu_seqlens_q[s+1]-cu_seqlens_q[s] and
 * k_len = cu_seqlens_k[s+1]-cu_seqlens_k[s] (0 <= q_len <= k_len), query i
 * (0-based) of head h attends to keys j <= i + (k_len - q_len) of KV head
 * h / (num_heads / num_kv_heads), read from the pool through block_tables[s].
 * The new tokens' K/V must already be in the pool (pkv_store_kvcache first),
 * so one call serves prompts with and without a cached prefix.
 *
 *   q    bf16 [total_q, num_heads, head_dim] packed
 *   out  bf16 [total_q, num_heads, head_dim] packed, written; rows of a
 *        sequence with q_len = 0 do not exist
 *   max_seqlen_q / max_seqlen_k  bounds on q_len / k_len (host-known)
 *   softmax_scale  > 0
 *   workspace  >= pkv_prefill_workspace_size(num_seqs, num_heads, num_kv_heads,
 *        head_dim, max_seqlen_q) bytes, 16-byte aligned: the work list, sorted
 *        by cost, that a planning launch writes before the attention launch
 *        reads it; needs no initialisation.  A sequence whose query rows fall
 *        outside [0, total_q), or whose lengths break the bounds above, is left
 *        out of the list and PKV_DEVERR_SEQLENS recorded.
 * Accumulation in fp32, probabilities rounded to bf16 for the PV product,
 * output rounded to bf16 once.
 */
PKV_API size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seqlen_q);

PKV_API pkv_status pkv_prefill_varlen(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                              int32_t max_seqlen_k, int32_t num_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, int32_t num_blocks,
                              float softmax_scale, pkv_bf16 *out, void *workspace,
                              size_t workspace_bytes, pkv_stream_t stream);

/*
 * a3, planned once per batch.  The engine prepares a step's inputs (cu_seqlens,
 * block tables) once, before the model runs (Nano-vLLM overview, the component
 * table: the model runner's prepare_prefill, then run), and every layer's
 * attention reads the same ones, so the work list can be made once and used by
 * every layer:
 *
 *   pkv_prefill_plan     writes the cost-sorted work list into workspace (one
 *                        small launch); it reads only cu_seqlens_q/k.
 *   pkv_prefill_varlen_planned
 *                        the attention of pkv_prefill_varlen, same arguments
 *                        and result, without the planning launch.
 *
 * A planned call must get the num_seqs, total_q, max_seqlen_k, group size
 * (num_heads / num_kv_heads), max_blocks_per_seq and block_size the plan was
 * made with, and cu_seqlens_q/k must hold the same values.  The plan carries a
 * tag of those arguments; a call whose arguments do not match it computes
 * nothing and records PKV_DEVERR_PLAN.  Each call leaves the workspace ready for
 * the next one, so any number of calls (each layer's pools, q and out) may
 * follow one plan, in order on one stream; two calls on one workspace must not
 * run at the same time.  A plan is valid until the workspace is reused for
 * anything else; pkv_prefill_varlen also leaves a plan for its own arguments.
 * Errors as for pkv_prefill_varlen (the plan checks only the arguments it takes).
 */
PKV_API pkv_status pkv_prefill_plan(const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            int32_t max_blocks_per_seq, int32_t num_seqs, int32_t total_q,
                            int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void *workspace,
                            size_t workspace_bytes, pkv_stream_t stream);

PKV_API pkv_status pkv_prefill_varlen_planned(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                      const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, int32_t num_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                      float softmax_scale, pkv_bf16 *out, void *workspace,
                                      size_t workspace_bytes, pkv_stream_t stream);

/*
 * a4. Decode attention: one query token per sequence over its whole context.
 * Visual atlas fig. 21 ("a decode step's real work": the newest token's KV is
 * written, then attention runs over the history); Nano-vLLM overview,
 * Sequence counters ([A,B,C] -> D): context_lens[b] counts every key the step
 * attends to, including the token whose KV this step wrote.
 *
 * out[b, h] = softmax_j(scale * q[b,h] . k_j) v_j over j < context_lens[b],
 * K/V head h / (num_heads / num_kv_heads), keys walked through
 * block_tables[b].  A sequence with context_lens[b] == 0 gets a zero row.
 *
 *   q    bf16 [batch, num_heads, head_dim];  out bf16 [batch, num_heads, head_dim]
 *   max_context_len  bound on context_lens (host-known); larger entries are
 *        clamped to max_blocks_per_seq * block_size and PKV_DEVERR_SEQLENS recorded
 *   workspace  >= pkv_decode_workspace_size(batch, num_heads, num_kv_heads,
 *        head_dim) bytes on the current device, 256-byte aligned; its contents
 *        need no initialisation and are scratch after the call
 * batch <= 4096 (PKV_ERR_UNSUPPORTED above, before any launch).
 * The work is split over the GPU's warps into equal runs of KV; partial
 * softmax states are merged in a fixed order, so results are deterministic.
 * softmax_scale must be a positive finite number (PKV_ERR_INVALID_ARG).
 */
PKV_API size_t pkv_decode_workspace_size(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                 int32_t head_dim);

PKV_API pkv_status pkv_decode(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *context_lens, int32_t batch, int32_t max_context_len,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t num_blocks, float softmax_scale,
                      pkv_bf16 *out, void *workspace, size_t workspace_bytes,
                      pkv_stream_t stream);

/*
 * a1 + a2 + a4 in one call: the decode step with the KV write fused in.
 * Visual atlas fig. 21 (the newest token's KV is written, then attention runs
 * over the whole history) and the offline explainer's scope box (input tokens
 * write KV first); slot rule of the atlas slot figure.
 *
 * For each sequence b with L = context_lens[b] > 0: the row of position L - 1
 * (slot = block_tables[b][(L-1) / bs] * bs + (L-1) % bs) of every KV head
 * receives k_new[b] / v_new[b], then out[b] is pkv_decode's result over the L
 * keys, now including that row.  Same result as pkv_slot_mapping (context_lens
 * form) + pkv_store_kvcache + pkv_decode, in two launches instead of four: the
 * warp that loads a sequence's last KV chunk writes the new row first.
 *
 *   k_new, v_new  bf16 [batch, num_kv_heads, head_dim], contiguous
 *   k_cache, v_cache  written at the new rows and read
 *   slot_mapping  int32 [batch] output, or NULL: each new token's slot (-1 for
 *                 a sequence with context_lens[b] == 0, which writes nothing)
 *   workspace     as for pkv_decode
 * A block id outside the pool skips the write and records PKV_DEVERR_BLOCK_ID.
 */
PKV_API pkv_status pkv_decode_append(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                             pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                             int32_t max_context_len, int32_t num_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, int32_t num_blocks,
                             float softmax_scale, pkv_bf16 *out, int32_t *slot_mapping,
                             void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * Decode without any allocation.  No step of the engine calls for it: this is a
 * library convenience for callers that cannot call cudaMalloc -- for example
 * a plugin inside a host runtime that owns all device memory and hands it only
 * its input and output buffers, or a service whose device-memory budget is
 * fixed at start-up.
 *
 * Same arguments and result as pkv_decode, minus the workspace: the scratch
 * is a PKV_DECODE_NOALLOC_SCRATCH_BYTES (4 MiB) array inside the library,
 * which every GPU that loads the library holds until the process exits.  A
 * batch whose pkv_decode_workspace_size() exceeds it returns
 * PKV_ERR_UNSUPPORTED (it fits up to 427 sequences with 8 KV heads on a
 * 152-SM GPU).
 * The first call on each device looks up the array's device address; make
 * that first call before any stream capture.  The address is kept for the
 * process: after a cudaDeviceReset this entry point must not be called again
 * (the same holds for every call of the library, whose per-device error word
 * and kernel set-up are kept the same way).  All calls share the array and
 * it keeps the last call's contents (nothing in it needs to start at zero);
 * calls that overlap on the GPU race on it and must be serialised.
 */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)

PKV_API pkv_status pkv_decode_noalloc(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *context_lens, int32_t batch, int32_t max_context_len,
                              int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t num_blocks, float softmax_scale,
                              pkv_bf16 *out, pkv_stream_t stream);

/*
 * a5. Temperature sampling by exponential race.
 * Visual atlas fig. 23: the engine samples with temperature only, as an
 * exponential race: winner = argmax_v p_v / e_v (= argmin e_v / p_v), with
 * p = softmax(logits / T) and e_v ~ Exp(1); not argmax p.
 *
 * Noise (the pages leave the generator open): Philox4x32-10 (Salmon et al.,
 * SC'11) with key (seed low 32, seed high 32) and counter (v / 4, row + offset
 * low 32, (row + offset) >> 32, 0); word v % 4 = x gives
 * u = (2 (x >> 9) + 1) 2^-24 and e_v = -ln u.  Since argmax p_v / e_v equals
 * argmax (logits_v / T - ln e_v), the kernel evaluates that form in fp32 in a
 * single pass over the logits; ties go to the lowest index.
 *
 *   logits        fp32 [batch, vocab], row b at logits + b * row_stride
 *   temperatures  fp32 [batch], each > 0
 *   out_ids       int64 [batch]; -1 for a row with an invalid temperature
 *                 (PKV_DEVERR_TEMPERATURE recorded) or no finite logit
 */
PKV_API pkv_status pkv_sample(const float *logits, int32_t batch, int32_t vocab, int64_t row_stride,
                      const float *temperatures, uint64_t seed, uint64_t offset,
                      int64_t *out_ids, pkv_stream_t stream);

/*
 * pkv_sample with the noise seed and row offset read from DEVICE memory:
 * seed_offset = uint64 [2] = {seed, offset}, 8-byte aligned, read when the
 * kernel runs.  A captured CUDA graph can then replay the sampler with fresh
 * noise by updating that buffer between replays (atlas fig. 26: a replay
 * reads new inputs from pre-allocated buffers).  Same result as pkv_sample
 * with those values.
 */
PKV_API pkv_status pkv_sample_dev(const float *logits, int32_t batch, int32_t vocab, int64_t row_stride,
                          const float *temperatures, const uint64_t *seed_offset, int64_t *out_ids,
                          pkv_stream_t stream);

/*
 * Read (and optionally clear) the current device's error word.  HOST output
 * pointers.  Synchronises the device.  code = PKV_DEVERR_*; info = a value
 * describing where (e.g. the sequence or token index).
 */
PKV_API pkv_status pkv_get_device_error(int32_t *code, int32_t *info, int32_t clear);

/*
 * Failure-path check.  Launches one CTA that waits, through the same bounded
 * mbarrier wait every kernel here uses, on a barrier that nothing completes.
 * The wait gives up after its limit (2 s), records PKV_DEVERR_TIMEOUT with
 * info PKV_WAIT_CHECK_INFO in the device error word, and the kernel returns:
 * no trap and no fault, so the context stays usable.  Asynchronous on
 * `stream`; read the result with pkv_get_device_error().
 */
#define PKV_WAIT_CHECK_INFO 0x5741
PKV_API pkv_status pkv_check_wait_timeout(pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
