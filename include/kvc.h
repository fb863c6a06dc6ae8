/*
 * kvc.h -- C ABI of libkvc, a paged KV cache and its decode step on NVIDIA
 * GB300 (sm_103a).
 *
 * What is computed follows three pages:
 *   "KV cache: Generation state, latency, and allocation" (aisyseng.dev,
 *   chapter 21), "KV Cache Explained: The Memory Problem Behind Fast LLM
 *   Inference" (archcrux.com) and the xf_kv_cache page (aicassindra.com).
 * Each entry point names the passage that defines its operation.
 *
 * Conventions for every call
 *   - Pointers marked "device" are caller-owned CUDA device memory of the
 *     pool's device; the library never frees them and keeps none after the
 *     call returns.  The pool owns its own device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously on it; the status reports argument validation
 *     and launch errors synchronously.  Problems that only the device can see
 *     (a table entry outside the pool, a position past its table row, a
 *     bounded wait that expired) never fault the GPU: the kernel skips the
 *     access and records an error bit, returned by kvc_pool_sync_status.
 *   - Calls on one pool share its workspace and error word: order them on one
 *     stream (or serialise them).  A call made while the device is current
 *     on another GPU than the pool's returns KVC_ERR_ARG.
 *   - Block tables are int32 [B][max_blocks], row-major; entry j of row b is
 *     the physical block holding positions [j*bs, (j+1)*bs) of sequence b, or
 *     -1 when none is allocated.  One table serves every layer (a block id
 *     names the same block in every layer's region).
 *
 * Pool layout in HBM (layout version 1): one allocation; layer l, physical
 * block p, keys (kv = 0) or values (kv = 1), KV head h, slot s, channel c is
 * the element at index
 *        ((((l * N + p) * H_KV + h) * 2 + kv) * bs + s) * d_h + c
 * of bf16 (2 bytes) or e4m3 (1 byte) elements.  The keys and values of one
 * (layer, block, head) are therefore one contiguous run of 2*bs*d_h elements
 * (8 KiB for bs 16, d_h 128, bf16), which the decode kernel moves with one
 * tensor-memory-accelerator copy per 128-byte column band.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stdint.h>

#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvc_pool kvc_pool;   /* opaque; owns its device memory */
typedef void *kvc_stream_t;         /* a cudaStream_t */

typedef enum {
    KVC_BF16 = 0,       /* 2-byte bfloat16 elements, stored bit for bit */
    KVC_FP8_E4M3 = 1,   /* 1-byte OCP E4M3 ("FN") elements with fp32 per-(head, channel) scales */
    KVC_INT4 = 2        /* 4-bit elements, q = rint(x / scale) in [-7, 7] stored as q + 8, two per byte
                         * (even channel in the low nibble), fp32 per-(head, channel) scales
                         * (the xf_kv_cache page: "int4 with per-channel scales") */
} kvc_dtype;

typedef enum {
    KVC_OK = 0,
    KVC_ERR_ARG = 1,          /* invalid argument (null pointer, shape, layer, misaligned pointer, wrong device) */
    KVC_ERR_OOM = 2,          /* device allocation failed */
    KVC_ERR_BAD_BLOCK = 3,    /* a table entry read by the kernel is -1 or >= num_blocks (device-detected) */
    KVC_ERR_RANGE = 4,        /* a position lies past its table row, or a length is negative (device-detected) */
    KVC_ERR_ALIAS = 5,        /* a write into a block other sequences still map (kvc_alloc_commit); the
                               * device calls do not detect aliasing: see kvc_decode_step */
    KVC_ERR_STALE = 6,        /* a lease stamp no longer current: the sequence was released or one of its
                               * table entries was replaced (kvc_alloc_check) */
    KVC_ERR_TIMEOUT = 7,      /* a bounded device-side wait expired (2 s); results of that call are invalid.
                               * The environment variable KVC_TEST_STALL (a test hook) withholds every
                               * call's copies so that its waits expire */
    KVC_ERR_CUDA = 8,         /* a CUDA runtime call failed */
    KVC_ERR_UNSUPPORTED = 9   /* a valid shape this build has no kernel for (see each call) */
} kvc_status;

/* Pool description returned by kvc_pool_info. */
typedef struct {
    int32_t layout_version;         /* 1: the index formula above */
    int32_t block_size;             /* bs, positions per block */
    int32_t num_layers;             /* L */
    int32_t num_kv_heads;           /* H_KV */
    int32_t head_dim;               /* d_h */
    int32_t dtype;                  /* kvc_dtype */
    int32_t elem_bytes;             /* s: 2 (bf16), 1 (e4m3), 0 (int4: half a byte, see elem_bits) */
    int32_t device;                 /* CUDA ordinal the pool lives on */
    int64_t num_blocks;             /* N */
    uint64_t block_bytes_per_layer; /* 2 * H_KV * bs * d_h * s */
    uint64_t layer_bytes;           /* N * block_bytes_per_layer */
    uint64_t bytes_per_token;       /* 2 * L * H_KV * d_h * s  ("KV Cache Explained", per-token size) */
    uint64_t capacity_tokens;       /* N * bs */
    uint64_t pool_bytes;            /* L * layer_bytes */
    void *base;                     /* device pointer of element 0 */
    float *scales;                  /* device fp32 [L][2][H_KV][d_h] (keys first) for e4m3 / int4 pools, else NULL */
    int32_t elem_bits;              /* 16, 8 or 4 */
    int32_t reserved;
} kvc_pool_desc;

/* ------------------------------------------------------------------ pool */

/* Allocate a pool of `num_blocks` fixed-size physical blocks of `block_size`
 * positions for `num_layers` layers on the current device
 * ("KV cache: Generation state, latency, and allocation" 21.5: fixed-size
 * blocks allocated as sequences grow; "KV Cache Explained", "Why
 * PagedAttention allocates KV in blocks": the pool is initialised up front).
 * Bytes: L * N * 2 * H_KV * bs * d_h * s (s = 1/2 for int4), plus for e4m3 / int4 the scale array
 * (initialised to 1.0).  Pool contents are uninitialised.
 * Limits: 1 <= block_size <= 128, head_dim 64 or 128 for bf16 and 128 for
 * e4m3 and int4 (the widths the attention kernels serve), 1 <= H_KV <= 256,
 * num_blocks >= 1, the pool's total row count L*N*H_KV*2*bs < 2^31.
 * Every attention call (kvc_decode_attn, kvc_decode_step, kvc_prefill_attn,
 * kvc_mixed_step, kvc_decode_attn_noalloc) needs block_size 16; a pool of
 * another block size serves kvc_append, kvc_write_tokens and kvc_copy_blocks
 * (e.g. the 4-position blocks of Table 21.1) and its attention calls return
 * KVC_ERR_UNSUPPORTED.  Errors: KVC_ERR_ARG, KVC_ERR_OOM, KVC_ERR_CUDA; *out is
 * NULL on error. */
KVC_API kvc_status kvc_pool_create(int64_t num_blocks, int32_t block_size, int32_t num_layers,
                           int32_t num_kv_heads, int32_t head_dim, kvc_dtype dtype, kvc_pool **out);

/* Free the pool's device memory after synchronising the device.  NULL is a no-op. */
KVC_API void kvc_pool_destroy(kvc_pool *pool);

/* Fill *desc.  Errors: KVC_ERR_ARG for NULL arguments. */
KVC_API kvc_status kvc_pool_info(const kvc_pool *pool, kvc_pool_desc *desc);

/* Set layer `layer`'s e4m3 scales: s_k, s_v are device fp32 [H_KV][d_h]
 * ("KV Cache Explained", "What changes when you use FP8 KV": quantized values
 * need scales; per-(KV head, channel) granularity), e4m3 or int4 pools.
 * Stored as given; a scale must be a positive finite float.  Errors: KVC_ERR_ARG (bf16 pool,
 * layer out of range, NULL), KVC_ERR_CUDA. */
KVC_API kvc_status kvc_pool_set_scales(kvc_pool *pool, int32_t layer, const float *s_k, const float *s_v,
                               kvc_stream_t stream);

/* Calibrate layer `layer`'s scales from bf16 tokens: absmax over the given
 * positions per (KV head, channel), divided by 448 (the largest finite E4M3
 * value) for e4m3 pools or by 7 (the int4 range) for int4 pools, in fp32; a
 * channel whose absmax is 0 gets scale 1.
 * k, v: device bf16 [n_tokens][H_KV][d_h].  With accumulate = 0 the running
 * absmax is reset first; with accumulate = 1 it extends the previous calls',
 * so a context uploaded in pieces calibrates like one array.  The scales are
 * rewritten after every call.  Errors: KVC_ERR_ARG, KVC_ERR_CUDA. */
KVC_API kvc_status kvc_calibrate_scales(kvc_pool *pool, int32_t layer, const void *k, const void *v,
                                        int64_t n_tokens, int32_t accumulate, kvc_stream_t stream);
/* The same call under its first name (e4m3 pools). */
KVC_API kvc_status kvc_calibrate_fp8(kvc_pool *pool, int32_t layer, const void *k, const void *v,
                             int64_t n_tokens, int32_t accumulate, kvc_stream_t stream);

/* ------------------------------------------------------------------ append */

/* Append one processed token per sequence at one layer
 * ("KV cache: Generation state, latency, and allocation" Eq. 21.6,
 * cache_t = append(cache_{t-1}, K_t, V_t), and Table 21.1 steps 1-2).
 * Sequence b's new key and value are written at position t = seq_lens[b]:
 * physical block block_tables[b][t / bs], slot t mod bs.  bf16 pools store
 * the bits unchanged; e4m3 pools store e4m3(fp32(k) / scale[h][c]) rounded to
 * nearest even and saturated to +-448.
 *   block_tables: device int32 [B][max_blocks]
 *   seq_lens:     device int32 [B], tokens held BEFORE the append (the write
 *                 position); the library never changes it
 *   k_new, v_new: device bf16 [B][H_KV][d_h], 4-byte aligned
 * The caller allocates block table[b][t / bs] before the call (the scheduler
 * owns allocation).  A token whose block entry is -1 / >= N, or whose
 * position is past the row, is skipped and recorded (KVC_ERR_BAD_BLOCK /
 * KVC_ERR_RANGE via kvc_pool_sync_status).  B = 0 is a no-op.
 * Errors (synchronous): KVC_ERR_ARG, KVC_ERR_CUDA. */
KVC_API kvc_status kvc_append(kvc_pool *pool, int32_t layer, const int32_t *block_tables, int32_t max_blocks,
                      const int32_t *seq_lens, int32_t B, const void *k_new, const void *v_new,
                      kvc_stream_t stream);

/* Write a ragged batch of tokens, e.g. a prompt's or a prefill chunk's keys
 * and values (same passage as kvc_append, repeated for consecutive
 * positions).  Sequence b receives rows cu_tokens[b] .. cu_tokens[b+1]-1 of
 * k and v at positions start_pos[b], start_pos[b]+1, ...
 *   cu_tokens: device int32 [B+1], non-decreasing prefix sums from 0
 *   start_pos: device int32 [B]
 *   max_tokens: host upper bound of cu_tokens[b+1]-cu_tokens[b] (grid size);
 *               rows beyond it are not written
 *   k, v: device bf16 [cu_tokens[B]][H_KV][d_h]
 * Same storage rule and error behaviour as kvc_append. */
KVC_API kvc_status kvc_write_tokens(kvc_pool *pool, int32_t layer, const int32_t *block_tables, int32_t max_blocks,
                            const int32_t *start_pos, const int32_t *cu_tokens, int32_t B, int32_t max_tokens,
                            const void *k, const void *v, kvc_stream_t stream);

/* ------------------------------------------------------------------ attention */

/* Paged decode attention at one layer
 * ("KV cache: Generation state, latency, and allocation" 21.1: the new query
 * reads the cached keys and its own new key, normalises the scores and mixes
 * the values; 21.5: attention follows the block table; padded or unfilled
 * slots are excluded; the xf_kv_cache page: GQA head sharing).
 * For each sequence b and query head hq, with h = hq / (H_Q / H_KV) and
 * n = seq_lens[b] positions (the appended token included):
 *   x_t = scale * <q[b][hq], K[b][t][h]>,  t < n
 *   out[b][hq] = sum_t softmax(x)_t V[b][t][h],   lse[b][hq] = ln sum_t exp(x_t)
 * computed in fp32 on tensor cores (bf16 or f16 operands, fp32 accumulation)
 * with a split-K online softmax and a log-sum-exp merge.  The last split CTA
 * of a (sequence, KV head) merges its partials in the same launch; when they
 * exceed 64 partial rows (query heads x splits, e.g. 32-head groups; the
 * KVC_MERGE_ROWS environment variable moves this limit, up to 4096) a second
 * launch on the same stream merges them.  For e4m3 and int4 pools the key
 * scales are folded into q and the value scales into the output.
 *   q:        device bf16 [B][H_Q][d_h], 4-byte aligned
 *   seq_lens: device int32 [B], positions attended (after the append);
 *             n = 0 gives out = 0 and lse = -inf
 *   out:      device fp32 [B][H_Q][d_h];  lse: device fp32 [B][H_Q] or NULL
 * Requires H_Q % H_KV == 0 (else KVC_ERR_ARG), block_size 16 and
 * H_Q / H_KV <= 32 (else KVC_ERR_UNSUPPORTED); head_dim is 64 or 128 (bf16)
 * or 128 (e4m3, int4), as kvc_pool_create admits.  Groups of 32 query heads
 * on d_h 128 bf16 or e4m3 pools (MQA) run on tensor-memory (tcgen05)
 * kernels: one CTA per SM streams 128-position tiles, with scores and
 * outputs in tensor memory (e4m3 codes widened to f16, exactly, on the way);
 * the environment variable KVC_TC=0 selects the split kernel for them too.
 * The pool's workspace for
 * split partials grows on first use with a larger batch (a cudaMalloc, so
 * make one call before capturing a CUDA graph; see kvc_pool_reserve).
 * Device-detected errors as for kvc_append; the affected sequence's outputs
 * are then zero.  Errors (synchronous): KVC_ERR_ARG, KVC_ERR_UNSUPPORTED,
 * KVC_ERR_OOM, KVC_ERR_CUDA. */
KVC_API kvc_status kvc_decode_attn(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                           const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens, int32_t B,
                           float *out, float *lse, float scale, kvc_stream_t stream);

/* One decode step at one layer in a single attention launch: kvc_append
 * followed by kvc_decode_attn ("KV cache: Generation state, latency, and allocation"
 * Eq. 21.6 and 21.1: the pass appends its token's key and value, and the new
 * query reads every cached key plus its own).  seq_lens holds the counts
 * BEFORE the append; sequence b's k_new/v_new rows are stored at position
 * seq_lens[b] exactly as kvc_append stores them, and attention runs over
 * seq_lens[b] + 1 positions.  The CTA that owns a sequence's last block
 * writes the new rows to the pool and into its staged copy of that block, so
 * the pool bytes and the outputs are bit-identical to the two separate calls.
 * The block receiving an append must not be mapped by another sequence of the
 * same call (shared blocks are copied before a write: 21.5, copy-on-write).
 *   k_new, v_new: device bf16 [B][H_KV][d_h], 16-byte aligned
 * Other arguments, requirements and errors as kvc_decode_attn. */
KVC_API kvc_status kvc_decode_step(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                                   const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens, int32_t B,
                                   const void *k_new, const void *v_new, float *out, float *lse, float scale,
                                   kvc_stream_t stream);

/* Causal attention of a prefill chunk over one sequence's paged cache
 * ("KV cache: Generation state, latency, and allocation" 21.3, chunked
 * prefill: later portions keep the earlier positions; the xf_kv_cache page,
 * "End-to-end flow": the new tokens attend to the shared prefix, the table
 * stitching shared and private blocks into one sequence).  Query i sits at
 * position q_start + i and reads positions 0 .. q_start + i, so its keys and
 * values must already be in the pool (kvc_write_tokens).  bf16 pools run on a
 * tensor-memory (tcgen05) kernel: 128 query rows (128 / g positions x the g
 * heads of a KV head) per CTA, scores and outputs in tensor memory (KVC_TC=0
 * selects the warp-level kernels).
 *   q: device bf16 [n_q][H_Q][d_h];  block_table_row: device int32 [max_blocks]
 *   out: device fp32 [n_q][H_Q][d_h];  lse: device fp32 [n_q][H_Q] or NULL
 * Same arithmetic, requirements and errors as kvc_decode_attn. */
KVC_API kvc_status kvc_prefill_attn(kvc_pool *pool, int32_t layer, const void *q, int32_t n_q, int32_t num_q_heads,
                            const int32_t *block_table_row, int32_t max_blocks, int32_t q_start,
                            float *out, float *lse, float scale, kvc_stream_t stream);

/* A decode step and a prefill chunk together ("KV cache: Generation
 * state, latency, and allocation" 21.3: chunked prefill runs beside the
 * decode steps of other requests; the xf_kv_cache page, "End-to-end flow").
 * Computes exactly what kvc_decode_step(q .. lse) followed by
 * kvc_prefill_attn(prefill_q .. prefill_lse) compute, with the chunk's work
 * running beside the decode step's so that its tensor-core work overlaps the
 * HBM stream: on bf16 pools the decode launch is followed by the
 * tensor-memory prefill kernel launched as its programmatic dependent (its
 * CTAs take SMs as the decode CTAs drain; it reads nothing the step writes
 * and never waits on it); on e4m3 and int4 pools one kernel's CTAs are the
 * two calls' CTAs interleaved.  The prefill row's positions
 * 0 .. q_start + n_q - 1 must already be in the pool and must not be among
 * the positions the decode part appends (they are written meanwhile).
 * n_q == 0 or B == 0 reduces to the other call alone.  On e4m3 and int4 pools,
 * decode groups of more than 16 query heads run the two calls in order.
 * Arguments, requirements and errors as kvc_decode_step and kvc_prefill_attn. */
KVC_API kvc_status kvc_mixed_step(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                                  const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens, int32_t B,
                                  const void *k_new, const void *v_new, float *out, float *lse,
                                  const void *prefill_q, int32_t n_q, const int32_t *prefill_block_table_row,
                                  int32_t prefill_max_blocks, int32_t q_start, float *prefill_out, float *prefill_lse,
                                  float scale, kvc_stream_t stream);

/* Pre-size the decode workspace for up to max_batch sequences of up to
 * max_blocks table entries and num_q_heads query heads, so that later
 * kvc_decode_attn / kvc_decode_step calls allocate nothing (a kvc_mixed_step
 * also needs counters for its chunk's query tiles: reserve with max_batch plus
 * the chunk's tiles, n_q / (64 / g) or n_q / (32 / g) rounded up, to cover it).
 * Errors: KVC_ERR_ARG, KVC_ERR_OOM. */
KVC_API kvc_status kvc_pool_reserve(kvc_pool *pool, int32_t max_batch, int32_t num_q_heads, int32_t max_blocks);

/* Decode attention that allocates no device memory.  The pages have no
 * counterpart to this call; it exists for callers that must not allocate in
 * the middle of a decode step: engines whose device memory is fully
 * pre-reserved by their own caching allocator (a cudaMalloc would fail or
 * fragment memory promised to KV blocks), and latency-critical loops where
 * cudaMalloc / cudaFree would synchronise the device and stall other streams.
 * Same arguments, arithmetic and results as kvc_decode_attn, but the split
 * partials live in a fixed 8 MiB device array inside the library instead of
 * the pool's workspace, so no cudaMalloc, cudaFree or allocating routine runs.
 * The array exists on every GPU where the library's device code is loaded,
 * from then until that context is destroyed; kvc_pool_create loads it, so it
 * is reserved when the first pool of a device is created.
 * Limit: when the batch is split, B * H_Q * splits * (d_h + 2) floats must fit
 * in 8 MiB (2^21 floats), where splits is the split count kvc_decode_attn
 * would choose; a larger request returns KVC_ERR_ARG before any launch.
 * The array's device address is looked up (cudaGetSymbolAddress with the
 * pool's device current) at pool creation and cached per CUDA context, so a
 * context created anew after a device reset gets a fresh lookup; a call in a
 * context where no pool was created does the lookup itself and should come
 * before any stream capture.  Every call on a device shares the one array,
 * and it keeps the last call's contents (nothing in it needs to start at
 * zero: every partial read is written by the same call first), so calls that
 * overlap on the GPU (other streams, other threads, other pools of the same
 * device) race and must be serialised by the caller. */
KVC_API kvc_status kvc_decode_attn_noalloc(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                                           const int32_t *block_tables, int32_t max_blocks,
                                           const int32_t *seq_lens, int32_t B, float *out, float *lse,
                                           float scale, kvc_stream_t stream);

/* ------------------------------------------------------------------ block allocator (host) */

/* Host-side block allocator that produces the block tables the calls above
 * consume ("KV cache: Generation state, latency, and allocation" 21.5 and
 * Table 21.1 steps 1-5; 21.4 prefix identity; "KV Cache Explained", "Why
 * PagedAttention allocates KV in blocks" and "Follow the 32 GiB pool until it
 * cannot allocate one more block").  Pure host code: no device memory, not
 * thread-safe (one caller at a time).
 *   - Blocks come from a FIFO free queue (initial order `free_order`, a
 *     permutation of [0, N), or ascending when NULL); when it is empty, the
 *     least recently released evictable cached block is reclaimed; when both
 *     are empty a reservation fails with KVC_ERR_OOM and changes nothing.
 *   - Every block has a reference count: one per sequence mapping it.
 *   - A sequence releases its references; a block at count 0 returns to the
 *     free queue, or (retain_cached = 1, and the block is a published full
 *     block) stays as an evictable cached entry that a prefix match revives.
 *   - Copy-on-write: a reservation whose next write lands in a shared, partly
 *     filled block maps a fresh block instead and reports the (old, new) pair,
 *     which the caller copies on the device (kvc_copy_blocks) before writing.
 * Sequence ids are small integers; a released id is reused by the next new
 * sequence (lowest first).  Errors: KVC_ERR_ARG for unknown ids or bad
 * sizes, KVC_ERR_OOM as above, KVC_ERR_ALIAS for a commit into a shared block. */
typedef struct kvc_alloc kvc_alloc;

KVC_API kvc_status kvc_alloc_create(int64_t num_blocks, int32_t block_size, const int32_t *free_order,
                                    int32_t retain_cached, kvc_alloc **out);
KVC_API void kvc_alloc_destroy(kvc_alloc *alloc);
/* A new, empty sequence. */
KVC_API kvc_status kvc_alloc_new_seq(kvc_alloc *alloc, int32_t *seq);
/* A new sequence sharing the first n_tokens positions of src (its blocks
 * gain a reference; a partly filled last block is shared until written). */
KVC_API kvc_status kvc_alloc_fork(kvc_alloc *alloc, int32_t src, int32_t n_tokens, int32_t *seq);
/* Make room for n_tokens more positions: map new blocks as the sequence
 * crosses block boundaries (Table 21.1 step 2), copy-on-write as above.
 * cow_pairs: host int32 [max_cow][2] (old, new); *n_cow receives 0 or 1. */
KVC_API kvc_status kvc_alloc_reserve(kvc_alloc *alloc, int32_t seq, int32_t n_tokens, int32_t *cow_pairs,
                                     int32_t max_cow, int32_t *n_cow);
/* Record that n_tokens more positions were written (after kvc_append /
 * kvc_write_tokens). */
KVC_API kvc_status kvc_alloc_commit(kvc_alloc *alloc, int32_t seq, int32_t n_tokens);
/* Drop the sequence's references (Table 21.1 steps 4-5). */
KVC_API kvc_status kvc_alloc_release(kvc_alloc *alloc, int32_t seq);
/* Register the identities h_i = hash(h_{i-1}, tokens_i), h_0 = hash(salt), of
 * the sequence's full blocks covering tokens[0, n_tokens) (21.4). */
KVC_API kvc_status kvc_alloc_publish(kvc_alloc *alloc, int32_t seq, const int32_t *tokens, int32_t n_tokens,
                                     uint64_t salt);
/* A new sequence mapping the longest run of published full blocks whose
 * identities match tokens (same salt, exact token ids: a hash collision is a
 * miss); *hit_tokens = positions covered. */
KVC_API kvc_status kvc_alloc_match(kvc_alloc *alloc, const int32_t *tokens, int32_t n_tokens, uint64_t salt,
                                   int32_t *seq, int32_t *hit_tokens);
KVC_API kvc_status kvc_alloc_seq_info(const kvc_alloc *alloc, int32_t seq, int64_t *len, int32_t *n_blocks);
/* Host block-table rows (int32 [n][max_blocks], -1 padded) and lengths of the given sequences. */
KVC_API kvc_status kvc_alloc_block_tables(const kvc_alloc *alloc, const int32_t *seqs, int32_t n, int32_t max_blocks,
                                          int32_t *table, int32_t *lens);
KVC_API kvc_status kvc_alloc_counts(const kvc_alloc *alloc, int64_t *n_free, int64_t *n_used, int64_t *n_cached);
/* Lease stamps ("KV Cache Explained", "The lease race when KV crosses
 * workers": a party that hands a request's blocks to another must let the
 * receiver detect that the lease expired and the blocks may have gone to
 * another request -- generation checks, with a mismatch treated as failure).
 * kvc_alloc_lease returns an opaque stamp of the sequence's current table: it
 * changes when the sequence is released (its id may then be handed out again
 * and its blocks to other requests) and when copy-on-write replaces one of its
 * table entries; blocks mapped at the end of the table leave earlier stamps
 * valid (the entries they cover are unchanged).  kvc_alloc_check returns
 * KVC_OK if `stamp` is still current and KVC_ERR_STALE otherwise; a consumer
 * checks before it uses a table it received (e.g. before a decode step on a
 * transferred request).  Errors: KVC_ERR_ARG for an id never handed out (check)
 * or not live (lease). */
KVC_API kvc_status kvc_alloc_lease(const kvc_alloc *alloc, int32_t seq, uint64_t *stamp);
KVC_API kvc_status kvc_alloc_check(const kvc_alloc *alloc, int32_t seq, uint64_t stamp);
/* Reference count of a block, or -1 for an id outside the pool. */
KVC_API int32_t kvc_alloc_refcount(const kvc_alloc *alloc, int32_t block);

/* Device copy of whole blocks, every layer, keys and values (the copy of
 * copy-on-write, "KV cache: ..." 21.5).  pairs: device int32 [n][2] (src, dst).
 * An id outside the pool is skipped and recorded (KVC_ERR_BAD_BLOCK via
 * kvc_pool_sync_status).  Errors: KVC_ERR_ARG, KVC_ERR_CUDA. */
KVC_API kvc_status kvc_copy_blocks(kvc_pool *pool, const int32_t *pairs, int32_t n, kvc_stream_t stream);

/* ------------------------------------------------------------------ host utilities */

/* Ideal KV payload in bytes
 * ("KV cache: Generation state, latency, and allocation" Eq. 21.2):
 * 2 * L * B * H_KV * T * d_h * s.  Pure host arithmetic, exact in uint64;
 * returns UINT64_MAX if an argument is negative or the product overflows. */
KVC_API uint64_t kvc_bytes(int64_t L, int64_t B, int64_t H_KV, int64_t T, int64_t d_h, int64_t s);

/* Wait for `stream`, then return and clear the pool's device-detected error
 * bits (the first of BAD_BLOCK, RANGE, TIMEOUT that is set), or KVC_OK.  A
 * CUDA error seen while waiting returns KVC_ERR_CUDA. */
KVC_API kvc_status kvc_pool_sync_status(kvc_pool *pool, kvc_stream_t stream);

/* Static description of a status code. */
KVC_API const char *kvc_status_str(kvc_status status);

/* Kernels this library has launched in this process (all pools, all devices). */
KVC_API uint64_t kvc_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
