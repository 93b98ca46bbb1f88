/*
 * paged_decode_attn.h - C ABI of the GB300 (sm_103a) paged MQA/GQA
 * decode-attention library.
 *
 * The operation (Loom Kernels landing page, "Supported now": "Paged MQA/GQA
 * decode", GQA packing + local split-K/LSE; benchmark page, "Current
 * qualified results": the D128 long-context split-K/LSE path). For every
 * sequence b < batch and query head hq < Hq, with G = Hq / Hkv, kv head
 * h = hq / G and L = context_lens[b]:
 *
 *   k_t = k_cache[block_table[b, t / block_size], t % block_size, h, :]   t < L
 *   v_t = v_cache[block_table[b, t / block_size], t % block_size, h, :]
 *   out[b, hq, :] = sum_t softmax_t(scale * q[b, hq, :] . k_t) * v_t
 *
 * The G query heads of one kv head are processed together against a single
 * read of that head's K/V pages (GQA packing). Long contexts are cut along
 * the sequence into page-aligned splits (split-K); each split yields a
 * normalised partial output and its log-sum-exp, and the splits are merged
 * by log-sum-exp weighting. Accumulation is in fp32.
 *
 * Conventions (Loom Kernels landing page, "Architecture": one versioned,
 * panic-contained framework boundary; borrowed streams and memory; explicit
 * layouts, aliasing rules and capabilities):
 *   - every function returns a pda_status (or a value documented below) and
 *     never throws, aborts or exits; on failure the reason is kept in a
 *     thread-local string returned by paged_decode_attn_last_error();
 *   - all tensors are caller-owned DEVICE memory, borrowed for the duration
 *     of the launch; the handle owns only its split-K workspace;
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream); run calls are asynchronous on it and never synchronise,
 *     allocate or read device memory from the host;
 *   - layouts are dense and row-major exactly as written below; element
 *     counts are int64-safe;
 *   - only `out` is written; it must not overlap q, k_cache, v_cache,
 *     block_table or context_lens (PDA_EALIAS). Repeated entries inside
 *     block_table (shared prefix pages) are legal;
 *   - one handle must not be used by two streams at the same time: the
 *     split-K workspace is per handle.
 *
 * Preconditions the host cannot check (device-resident values), and what
 * happens when they are broken:
 *   - 0 <= context_lens[b] <= max_blocks * block_size: larger values are
 *     clamped to max_blocks * block_size, negative values act as 0;
 *   - 0 <= block_table[b, p] < num_blocks for p < ceil(L / block_size):
 *     out-of-range ids read zeros (the tensor-memory-access unit bounds-checks
 *     every page fetch); entries at p >= ceil(L / block_size) are never read;
 *   - a row with L == 0 is written as zeros.
 *   paged_decode_attn_validate() reports broken preconditions without
 *   faulting.
 */
#ifndef PAGED_DECODE_ATTN_H
#define PAGED_DECODE_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PDA_ABI_VERSION 2

typedef enum {
  PDA_OK = 0,
  PDA_EINVAL = -1,       /* bad argument (null pointer, shape, size limit) */
  PDA_EUNSUPPORTED = -2, /* valid but not built: head_dim, group size, block size */
  PDA_ENOMEM = -3,       /* workspace allocation failed in create */
  PDA_ECUDA = -4,        /* a CUDA runtime/driver call failed (message says which) */
  PDA_EALIAS = -5,       /* out overlaps an input */
  PDA_EDEVICE = -6       /* the device reported an error word (see check_device_error) */
} pda_status;

typedef enum {
  PDA_BF16 = 0,
  PDA_FP16 = 1,
  PDA_F32 = 2 /* output only: fp32 out for accuracy checks */
} pda_dtype;

/* Fixed at create time. Supported geometries: G = Hq / Hkv from 1 to 16 at
 * head_dim 64 or 128 (G 9..16 on the tensor-core kernel only), 1 to 4 at
 * head_dim 256; with kv_fp8, any G up to 16 at head_dim 64 or 128 and dtype
 * PDA_BF16 or PDA_FP16. */
typedef struct {
  int num_q_heads;        /* Hq; a multiple of num_kv_heads */
  int num_kv_heads;       /* Hkv */
  int head_dim;           /* D; 64, 128 or 256 */
  int block_size;         /* tokens per page; 16 or 32, or 64 at G <= 8 */
  int dtype;              /* pda_dtype of q and out (and of the caches unless kv_fp8):
                             PDA_BF16 or PDA_FP16 */
  int max_batch;          /* largest batch a run may pass (1 .. 65535) */
  int max_blocks_per_seq; /* largest max_blocks a run may pass */
  int max_splits;         /* largest split count (1 .. 64); sizes the workspace */
  int device;             /* CUDA device ordinal the handle and its launches use */
  int kv_fp8;             /* 0: k_cache/v_cache hold dtype values; 1: they hold FP8 E4M3
                             bytes (OCP "e4m3fn": bias 7, no infinities, max 448) that
                             paged_decode_attn_run_scaled dequantises with per-kv-head
                             scales (landing page, "Next boundaries": FP8 KV-cache
                             compression) */
} pda_config;

typedef struct pda_handle_s* pda_handle;

/* PDA_ABI_VERSION of the loaded library. */
int paged_decode_attn_abi_version(void);

/* Thread-local description of the last failure on this thread ("" if none).
 * The pointer stays valid until the next call on the same thread. */
const char* paged_decode_attn_last_error(void);

/* Validate `cfg`, select cfg->device, and allocate the handle plus its
 * device workspace: max_batch * Hq * max_splits * (head_dim + 1) floats of
 * split partials, max_batch * Hkv ints of split tickets (the last split of a
 * sequence's kv head to finish merges the splits; tickets return to zero by
 * the end of every call) and a small error-word area, all zeroed.
 * Returns PDA_OK and stores the handle in *out_handle, or an error (and
 * *out_handle = NULL). Configuration errors are reported before any CUDA call. */
int paged_decode_attn_create(const pda_config* cfg, pda_handle* out_handle);

/* Release the handle and its workspace. NULL is a no-op. The caller must
 * make sure no launch using the handle is still running. */
void paged_decode_attn_destroy(pda_handle handle);

/* Paged decode attention for one decode step.
 *   q            [batch, Hq, D]                          cfg->dtype
 *   k_cache      [num_blocks, block_size, Hkv, D]        cfg->dtype
 *   v_cache      [num_blocks, block_size, Hkv, D]        cfg->dtype
 *   block_table  [batch, max_blocks]                     int32
 *   context_lens [batch]                                 int32
 *   out          [batch, Hq, D]                          cfg->dtype
 * batch <= cfg->max_batch (0 is a no-op), max_blocks <= cfg->max_blocks_per_seq,
 * num_blocks * block_size < 2^31; q, caches and out 16-byte aligned.
 * scale multiplies q . k (typically 1/sqrt(D)); it must be finite.
 * The split count comes from the built-in heuristic (paged_decode_attn_plan). */
int paged_decode_attn_run(pda_handle handle, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_table,
                          const int32_t* context_lens, int batch, int max_blocks,
                          int64_t num_blocks, float scale, void* out, void* stream);

/* As paged_decode_attn_run, plus:
 *   num_splits            0 = heuristic; otherwise the split count to use
 *                         (1 .. cfg->max_splits, clipped to the page count
 *                         implied by max_context_len_hint)
 *   max_context_len_hint  0 = max_blocks * block_size; otherwise the length
 *                         the planner sizes splits for. A longer sequence is
 *                         still exact: its last split takes the remaining
 *                         pages (less balanced, never wrong).
 *   out_dtype             PDA_F32 writes fp32 `out`; -1 or cfg->dtype writes
 *                         the input dtype (round to nearest even). */
int paged_decode_attn_run_ex(pda_handle handle, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* block_table,
                             const int32_t* context_lens, int batch, int max_blocks,
                             int64_t num_blocks, float scale, void* out, void* stream,
                             int num_splits, int max_context_len_hint, int out_dtype);

/* As paged_decode_attn_run_ex, with K/V dequantisation scales:
 *   k_t = k_scale[h] * k_cache[...],  v_t = v_scale[h] * v_cache[...]
 * for kv head h (scale_per_head = 1: arrays of Hkv fp32 values; 0: one fp32
 * value each, a per-tensor scale). Device pointers; NULL means 1. Any cache
 * type may be scaled; FP8 caches (cfg->kv_fp8) are 1-byte elements with the
 * same [num_blocks, block_size, Hkv, D] layout. */
int paged_decode_attn_run_scaled(pda_handle handle, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_table,
                                 const int32_t* context_lens, int batch, int max_blocks,
                                 int64_t num_blocks, float scale, const float* k_scale,
                                 const float* v_scale, int scale_per_head, void* out,
                                 void* stream, int num_splits, int max_context_len_hint,
                                 int out_dtype);

/* The split plan the heuristic picks (host only, no CUDA call): for a
 * problem of `batch` sequences, `max_blocks` table columns and an optional
 * length hint (0 = max_blocks * block_size), on a GPU with `num_sms` SMs.
 * *num_splits receives S (1 .. cfg->max_splits) and *chunk_pages the pages
 * each split covers; sequence b then uses min(S, ceil(ceil(L_b / block_size)
 * / chunk_pages)) splits. Waves of work units are counted over 27/32 of the
 * SMs for the 16-bit tensor-core kernel (G 3..16 at head_dim 64/128) and over
 * every SM (times CTAs per SM) otherwise. The kernel is chosen per call: a
 * call of 16-bit K/V at G <= 8 whose longest context L (max_blocks *
 * block_size, or the hint when smaller) and K/V bytes (at most batch * Hkv *
 * L * head_dim * 4) are small (L <= 256 and <= 48 MiB, or L <= 1024 and
 * <= 20 MiB) runs on the CUDA-core kernel, where the tensor-core kernel's
 * fixed cost would dominate. */
int paged_decode_attn_plan(const pda_config* cfg, int num_sms, int batch, int max_blocks,
                           int max_context_len_hint, int* num_splits, int* chunk_pages);

/* How paged_decode_attn_run_ex with these arguments is launched on this
 * handle's GPU (host only, no CUDA call): *splits and *chunk_pages as in
 * paged_decode_attn_plan (num_splits 0 = the heuristic), *ctas the CTAs of
 * the partial kernel, and *cluster the CTAs per thread-block cluster. With
 * the tensor-core kernel, a split count of 2..16 whose batch * Hkv
 * (sequence, kv head) pairs all fit on the GPU at once as clusters of that
 * many CTAs runs as one cluster per pair, one CTA per split, and the splits
 * merge through distributed shared memory (*cluster = splits); otherwise
 * *cluster = 1 and the last split of a pair merges through the handle's
 * workspace. (Landing page, "Supported now": split-K with log-sum-exp
 * merge; the cluster layout is this library's GB300 design.) */
int paged_decode_attn_launch_shape(pda_handle handle, int batch, int max_blocks,
                                   int max_context_len_hint, int num_splits, int* splits,
                                   int* chunk_pages, int* ctas, int* cluster);

/* Log-sum-exp merge of split partials (the split-K merge step on its own,
 * e.g. for partials computed elsewhere):
 *   partial_o   [rows, num_splits, head_dim] fp32, each split's normalised output
 *   partial_lse [rows, num_splits] fp32, natural-log sum of exp(scaled logits)
 *               of each split; -inf marks an empty split (weight 0)
 *   out         [rows, head_dim] in out_dtype (PDA_BF16, PDA_FP16 or PDA_F32)
 *   out[r] = sum_s exp(lse[r,s] - M) o[r,s] / sum_s exp(lse[r,s] - M),
 *   M = max_s lse[r,s]; a row of all-empty splits is written as zeros.
 * head_dim must be a multiple of 4 (<= 512), num_splits 1 .. 64; device pointers,
 * asynchronous on `stream`. No handle needed. */
int paged_decode_attn_merge(const float* partial_o, const float* partial_lse, int rows,
                            int num_splits, int head_dim, void* out, int out_dtype,
                            int device, void* stream);

/* Opt-in precondition check on device-resident inputs (asynchronous on
 * `stream`): flags context_lens[b] outside [0, max_blocks * block_size] and
 * block_table entries outside [0, num_blocks) among the pages a sequence
 * reads. It records the first problem found in the handle's device error
 * word; it never traps. Read it with paged_decode_attn_check_device_error. */
int paged_decode_attn_validate(pda_handle handle, const int32_t* block_table,
                               const int32_t* context_lens, int batch, int max_blocks,
                               int64_t num_blocks, void* stream);

/* Synchronise `stream`, read and clear the handle's device error word.
 * *code receives 0 (no error) or a nonzero code:
 *   1 = context length out of range, 2 = block id out of range (validator);
 *   3 = a pipeline wait inside a kernel gave up after its time limit.
 * (Codes 4 and 5 belong to the error words of paged_decode_attn_rope_kv_write and of
 * the KV-cache movement calls.)
 * *detail receives the sequence index (codes 1, 2) or the split index (3).
 * Returns PDA_OK, or PDA_ECUDA if the synchronisation or the copy failed. */
int paged_decode_attn_check_device_error(pda_handle handle, int* code, int* detail,
                                         void* stream);

/* RoPE + paged-KV write (Loom Kernels landing page, "Supported now": "RoPE +
 * paged-KV write", packed Q/K rotation + native cache write): rotates the
 * new tokens' query and key heads and stores key and value heads into the
 * paged cache read by paged_decode_attn_run, in one launch. No handle.
 *
 * For token t < num_tokens with p = positions[t] and table row
 * cs = cos_sin_cache[p] (rot_dim floats: rot_dim/2 cosines, then rot_dim/2
 * sines), every head vector x of q and k has its pairs j < rot_dim/2,
 *   (a, b) = (j, j + rot_dim/2)   neox_style != 0 (rotate halves)
 *   (a, b) = (2j, 2j + 1)         neox_style == 0 (interleaved pairs),
 * rotated as y_a = x_a cos_j - x_b sin_j, y_b = x_b cos_j + x_a sin_j; dims
 * >= rot_dim are copied. Outputs are exactly rounded (round to nearest even
 * of the double-precision value), so the result is bit-identical to the FP64
 * definition.
 *   q        [num_tokens, num_q_heads, head_dim], token stride q_token_stride
 *   k, v     [num_tokens, num_kv_heads, head_dim], token strides k/v_token_stride
 *            (strides in elements; 0 = packed; e.g. views into a fused qkv
 *            projection output)
 *   positions     [num_tokens] int32
 *   slot_mapping  [num_tokens] int64: cache row of the token
 *                 (block * block_size + offset in block); < 0 = no cache write
 *   cos_sin_cache [max_position, rot_dim] fp32 (may be NULL when rot_dim = 0)
 *   q_out    [num_tokens, num_q_heads, head_dim], token stride q_out_token_stride;
 *            q_out == q with equal strides rotates in place
 *   k_cache, v_cache  [num_slots, num_kv_heads, head_dim] (the decode
 *            layout [num_blocks, block_size, Hkv, D] with num_slots =
 *            num_blocks * block_size); only the rows named by slot_mapping
 *            are written
 *   err      optional device int[2] (NULL = none): the first bad token sets
 *            err[0] = 4 (position outside [0, max_position)) or 5 (slot >=
 *            num_slots) and err[1] = its index; the caller zeroes it.
 * A token with a bad position writes nothing; one with a bad slot writes
 * q_out only. Two tokens with the same slot race (last writer undefined).
 * dtype PDA_BF16 or PDA_FP16 for q, k, v, q_out and the caches; head_dim a
 * multiple of 16 (<= 1024), rot_dim a multiple of 16 (<= head_dim); every
 * pointer 16-byte aligned, token strides multiples of 8. Outputs must not
 * overlap inputs or each other (PDA_EALIAS), except q_out == q. Asynchronous
 * on `stream`; allocates nothing; graph-capturable. */
int paged_decode_attn_rope_kv_write(const void* q, int64_t q_token_stride, const void* k,
                                    int64_t k_token_stride, const void* v,
                                    int64_t v_token_stride, const int32_t* positions,
                                    const int64_t* slot_mapping, const float* cos_sin_cache,
                                    int max_position, int rot_dim, int neox_style,
                                    int num_tokens, int num_q_heads, int num_kv_heads,
                                    int head_dim, int dtype, void* q_out,
                                    int64_t q_out_token_stride, void* k_cache, void* v_cache,
                                    int64_t num_slots, int* err, int device, void* stream);

/* KV-cache movement (landing page, "Next boundaries": KV-cache movement -
 * block copy, gather, scatter and compact work for prefix reuse and
 * preemption). Caches are [num_blocks, block_size, Hkv, D] of any element
 * type and are moved as raw bytes, so results are exact copies. All pointers
 * are device memory, calls are asynchronous on `stream`, allocate nothing
 * and may be captured in a CUDA graph. `err` is an optional device int[2]
 * (NULL = none) that receives the first out-of-range id found: code 1
 * (a length above max_len), 2 (a block id outside [0, num_blocks)) or 5 (a
 * slot past the cache), and its index; such entries are skipped, never
 * dereferenced. Sizes in bytes must be multiples of 16 and buffers 16-byte
 * aligned (index arrays: their element size). */

/* For i < n_pairs (<= 65535): block pairs[2i+1] of k_cache and of v_cache
 * becomes a copy of block pairs[2i] (int64 pairs). block_bytes =
 * block_size * Hkv * D * element size. Destinations must be distinct and
 * must not also be sources (then the pairs' order does not matter; a
 * compaction's moves into free blocks satisfy this). */
int paged_decode_attn_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks,
                                  int64_t block_bytes, const int64_t* pairs, int n_pairs,
                                  int* err, int device, void* stream);

/* Gather: for each sequence b < batch (<= 65535), its tokens t < lens[b]
 * (int32; read through block_table [batch, max_blocks] int32) are copied in
 * order to rows cu_rows[b] + t of k_out / v_out ([rows, Hkv, D], row_bytes =
 * Hkv * D * element size each); cu_rows [batch] int64 holds each sequence's
 * first row (e.g. exclusive prefix sums of lens), and the outputs must hold
 * every row it implies. max_len >= every lens[b] (<= max_blocks *
 * block_size) sizes the grid; a longer length is flagged (code 1) and cut. */
int paged_decode_attn_gather_kv(const void* k_cache, const void* v_cache, int64_t num_blocks,
                                int block_size, int64_t row_bytes, const int32_t* block_table,
                                int max_blocks, const int32_t* lens, const int64_t* cu_rows,
                                int batch, int max_len, void* k_out, void* v_out, int* err,
                                int device, void* stream);

/* Scatter: row r < n_rows of k_rows / v_rows ([n_rows, Hkv, D], row_bytes
 * each) is copied to cache slot slot_mapping[r] (int64; slot = block *
 * block_size + offset, num_slots = num_blocks * block_size); slot < 0 skips
 * the row. Two rows with the same slot race. */
int paged_decode_attn_scatter_kv(const void* k_rows, const void* v_rows, int64_t n_rows,
                                 int64_t row_bytes, const int64_t* slot_mapping, void* k_cache,
                                 void* v_cache, int64_t num_slots, int* err, int device,
                                 void* stream);

/* In place: block_table[b, p] := new_id[block_table[b, p]] for b < batch and
 * the pages p < ceil(lens[b] / block_size) a sequence uses (entries past
 * them are left alone); new_id has num_blocks int32 entries. With
 * copy_blocks this is a compaction: move the live blocks, then remap. */
int paged_decode_attn_remap_table(int32_t* block_table, int batch, int max_blocks,
                                  const int32_t* lens, int block_size, const int32_t* new_id,
                                  int64_t num_blocks, int* err, int device, void* stream);

/* Decode attention for callers that cannot allocate device memory.
 * (No counterpart in the paper: this entry point exists for integration.)
 *
 * Who needs it: code that runs where cudaMalloc is off limits, for example
 * inside a host callback or another library's allocator-free region, or a
 * runtime that owns every byte of device memory through its own pool and
 * forbids allocations behind its back. paged_decode_attn_create allocates
 * the split-K workspace, so such callers cannot use a handle.
 *
 * This call takes the geometry directly (no handle) and allocates nothing:
 * the split-K partials live in one fixed scratch array of 8 MiB of fp32
 * partial outputs, 256 KiB of fp32 log-sum-exps and 256 KiB of split
 * tickets, built into the library and held on every GPU that loads it until
 * the process exits. The split count the heuristic picks is lowered until
 * the partials fit (batch * Hq * S * head_dim <= 2^21, batch * Hq * S <= 2^16,
 * and no splitting at all if batch * Hkv > 2^16); a sequence with a single
 * split needs no scratch. An explicit num_splits runs as
 * S = ceil(max_blocks / chunk) splits of chunk = ceil(max_blocks /
 * min(num_splits, max_blocks)) pages, as in paged_decode_attn_run_ex; if that
 * S is above 1 and does not fit, the call is rejected with PDA_EINVAL and the
 * message names S and the largest split count that fits. Each call clears the
 * tickets it uses.
 *
 * Set-up: the first call on a device looks up the scratch array's device
 * address and sets the kernels' shared-memory limits for that device; make
 * that first call before any stream capture. Later calls only launch.
 *
 * Sharing: every call on a device uses the same scratch and it keeps the
 * last call's contents. Calls that can overlap on the GPU (different
 * streams, or different host threads) race on it and give wrong results;
 * serialise them. Device-side pipeline timeouts are not reported by this
 * entry point (it has no error word the caller can read).
 *
 * Arguments are those of paged_decode_attn_run_ex, with the geometry of
 * pda_config (num_q_heads, num_kv_heads, head_dim, block_size, dtype) in
 * place of the handle, out in the input dtype, and `device` the CUDA
 * ordinal the pointers belong to. Same layouts, alignment, aliasing rules,
 * return codes and asynchrony. */
int paged_decode_attn_run_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, const int32_t* context_lens,
                                  int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int dtype, int max_blocks, int64_t num_blocks,
                                  float scale, void* out, int num_splits, int device,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_DECODE_ATTN_H */
