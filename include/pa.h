/*
 * pa.h -- C ABI of libpa.so: batch-invariant paged-KV attention over one flat
 * ragged step of a continuous-batching engine, for NVIDIA GB300 (sm_103a).
 *
 * The operations are the ones "P3: native paged-KV continuous-batching
 * sampler" (section Design, paged.py) specifies for its paged attention seam:
 * write the step's new K/V rows into per-layer [num_blocks, block_size, Hkv, D]
 * caches by slot mapping, then return [T, H, D] attention for decode rows and
 * causal prefill chunks, reading keys through an int32 [B, max_blocks] block
 * table with cu_seqlens_q and ctx_lens, with the KV split fixed per context
 * length and no atomics in any reduction (the TritonPagedAttention contract of
 * that section). "Numerics envelopes" (sections The contract and The
 * hierarchy, invariance.batch) gives the property every entry point keeps: a
 * row's output bits do not depend on which other rows share the step.
 *
 * Conventions
 *   - All tensor arguments are DEVICE pointers to contiguous row-major arrays
 *     owned by the caller; the library allocates no device memory and keeps
 *     no per-call state. All work is enqueued on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream). Results are valid once the stream
 *     reaches that point. Only pa_read_status synchronises.
 *   - Element type `dtype` applies to q, caches, new rows and out alike,
 *     except PA_FP8_E4M3: caches hold e4m3 codes (1 byte) under per-tensor
 *     scales while q, new rows and out are bf16.
 *   - ctx_lens[b] counts every key lane b attends AFTER this step's write, its
 *     own new rows included; row j (0-based) of a lane with q_len rows sits at
 *     absolute position ctx_lens[b] - q_len + j and attends keys 0..position.
 *   - Query head h reads kv head h / (H / Hkv) (blocked GQA map).
 *   - Supported: D in {64, 128}; block_size in {16, 32}; H % Hkv == 0 and
 *     1 <= H / Hkv <= 16; dtype PA_F32, PA_BF16 or PA_FP8_E4M3.
 *
 * Errors
 *   - Problems visible on the host (NULL pointers, unsupported geometry,
 *     negative sizes, workspace too small) return a pa_status code before any
 *     CUDA call is made.
 *   - Problems only visible on the device (a slot or block id out of range,
 *     a lane whose ctx exceeds its block-table row, q_len > ctx_len, malformed
 *     cu_seqlens_q, more splits than the workspace holds) set bits of the
 *     int32 device status word (PA_FLAG_*) with an atomic OR; the offending
 *     write is skipped or the offending lane's rows are left unspecified, and
 *     no kernel ever traps. `status` may be NULL (flags are then dropped).
 *   - Launch failures return PA_ERR_CUDA (cudaGetLastError after launch).
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, inconsistent sizes */
  PA_ERR_UNSUPPORTED = 2,   /* geometry or dtype outside the supported set    */
  PA_ERR_WORKSPACE = 3,     /* workspace NULL, misaligned or too small        */
  PA_ERR_CUDA = 4           /* a CUDA runtime call or launch failed           */
} pa_status;

/*
 * Element types.
 *   PA_F32       q, caches, new rows and out in fp32
 *   PA_BF16      all of them in bf16
 *   PA_FP8_E4M3  q, new rows and out in bf16; the caches hold float8 e4m3fn
 *                codes (1 byte: sign, 4 exponent bits with bias 7, 3 mantissa
 *                bits; S.1111.111 is NaN; largest finite 448) under one fp32
 *                scale per tensor, k_scale for the K cache and v_scale for the
 *                V cache: a code c stands for e4m3(c) * scale. New rows are
 *                quantised on write as RN-even(x / scale) with x / scale in
 *                fp32, finite overflow and infinities saturating to +-448.
 *                ("P3: native paged-KV continuous-batching sampler", Review
 *                (adversarial pass), kv_dtype: K/V are dequantised on read;
 *                fp8 KV without per-tensor scales is visibly lossy.)
 */
typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/*
 * Invariance modes of pa_attention_ex.
 *   PA_MODE_BATCH_INVARIANT  a row's output bits depend only on its own lane
 *                            (q, keys, ctx_len, q_len), never on the other
 *                            lanes of the step. Decode rows (q_len == 1) take
 *                            the split-KV path; bf16 lanes with q_len >= 2
 *                            take the tensor-core prefill path.
 *   PA_MODE_ROW_INVARIANT    additionally independent of the row's own
 *                            lane's q_len: every row, decode or prefill, takes
 *                            the split-KV path with the split partition of
 *                            its own key count (position + 1), so a row has
 *                            the same bits whether it arrives as a decode row,
 *                            inside a prefill chunk of any length, or again
 *                            on recompute after a prefix hit at any token
 *                            ("Numerics envelopes", Prefix hits resume at any
 *                            token; "P3: native paged-KV continuous-batching
 *                            sampler", Evidence, batch invariance under
 *                            chunk sizes 1, 2 and 64). fp32 and e4m3 steps
 *                            always behave this way.
 */
/*
 *   PA_MODE_REUSE_PLAN       a bit OR-ed into either mode (pass
 *                            (pa_mode)(PA_MODE_... | PA_MODE_REUSE_PLAN)):
 *                            the workspace already holds the split plan a
 *                            previous pa_attention_ex call on the same
 *                            stream built for this step -- the same B, T, H,
 *                            Hkv, D, block size, dtype, mode, max_q_len,
 *                            max_ctx_len and workspace size, and the same
 *                            cu_seqlens_q and ctx_lens contents -- so the
 *                            call does not build it again: the layers of one
 *                            step attend over the same lanes, and only the
 *                            first layer's call needs to plan ("P3: native
 *                            paged-KV continuous-batching sampler", Design:
 *                            one flat step description serves the whole
 *                            forward pass). Everything else (the write of
 *                            the new rows, q, the caches, block tables, out)
 *                            is this call's own. The library checks the
 *                            sizes on the device: on a mismatch it raises
 *                            PA_FLAG_PLAN_MISMATCH, writes no output (the
 *                            write of new rows still happens) and discards
 *                            the stored plan, so later reusing calls are
 *                            refused too until a call without the bit plans
 *                            again. Changed
 *                            contents of cu_seqlens_q / ctx_lens are not
 *                            detected: the caller must then plan again
 *                            (a call without the bit). Output bits are the
 *                            same with or without the bit.
 */
typedef enum {
  PA_MODE_BATCH_INVARIANT = 0,
  PA_MODE_ROW_INVARIANT = 1,
  PA_MODE_REUSE_PLAN = 0x100
} pa_mode;

/* Device status word bits. */
#define PA_FLAG_SLOT_RANGE   0x01  /* slot >= num_blocks * block_size: write skipped      */
#define PA_FLAG_BLOCK_RANGE  0x02  /* block-table entry outside [0, num_blocks)          */
#define PA_FLAG_CTX_RANGE    0x04  /* ctx_len < 0 or > max_blocks_per_seq * block_size    */
#define PA_FLAG_QLEN_RANGE   0x08  /* q_len > ctx_len                                     */
#define PA_FLAG_CU_SEQLENS   0x10  /* cu_seqlens_q not 0 .. T and non-decreasing (then any
                                      row, of any lane, may be left unwritten)            */
#define PA_FLAG_WORKSPACE    0x20  /* the step needs more splits than the workspace holds */
#define PA_FLAG_HOST_BOUND   0x40  /* a lane exceeds the host's max_q_len / max_ctx_len   */
#define PA_FLAG_TIMEOUT      0x80  /* a bounded wait inside a kernel gave up              */
#define PA_FLAG_OWNER_RANGE  0x100 /* KV-parallel key ranges not split-aligned / not a
                                      partition of the lane's keys: lane skipped          */
#define PA_FLAG_PLAN_MISMATCH 0x200 /* PA_MODE_REUSE_PLAN, but the workspace's plan was
                                      built for other sizes: no output written            */

/*
 * pa_write_kv -- scatter T new K/V rows into the caches.
 * ("P3: native paged-KV continuous-batching sampler", Design, paged.py:
 *  PagedKVCache copy-free append into (block, offset).)
 *
 *   k_new, v_new     [T, Hkv, D]               rows to store
 *   k_cache, v_cache [num_blocks, block_size, Hkv, D]
 *   slot_mapping     int64 [T]; row t goes to block slot / block_size, offset
 *                    slot % block_size. slot < 0 skips the row (padding);
 *                    slot >= num_blocks * block_size sets PA_FLAG_SLOT_RANGE
 *                    and skips it.
 * Bytes move unchanged (bit-exact). Slots within one call must be distinct
 * and must not name blocks another sequence also references (a shared block
 * is read-only); neither is checked. Caches must not alias the new rows.
 * Pointers must be 16-byte aligned.
 */
pa_status pa_write_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int32_t T, int32_t num_blocks,
                      int32_t block_size, int32_t Hkv, int32_t D, pa_dtype dtype,
                      int32_t* status, void* stream);

/*
 * pa_write_kv_scaled -- pa_write_kv for every element type, with the scales
 * of PA_FP8_E4M3 caches (k_scale, v_scale: finite and > 0; ignored for the
 * other types, whose bytes are copied unchanged). For PA_FP8_E4M3, k_new and
 * v_new are bf16 [T, Hkv, D] and each element lands in the cache as its
 * e4m3 code (see pa_dtype). pa_write_kv refuses PA_FP8_E4M3 with
 * PA_ERR_UNSUPPORTED (it has no scales).
 */
pa_status pa_write_kv_scaled(const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, const int64_t* slot_mapping, int32_t T,
                             int32_t num_blocks, int32_t block_size, int32_t Hkv, int32_t D,
                             pa_dtype dtype, float k_scale, float v_scale, int32_t* status,
                             void* stream);

/*
 * pa_attention_workspace_bytes -- device scratch pa_attention needs.
 * ("P3: native paged-KV continuous-batching sampler", Design, paged.py: the
 *  paged-attention kernel contract's fixed KV split per context length --
 *  the split partials of that split are what this scratch holds -- and
 *  PagedKVCache.ensure_capacity, all-or-nothing: the caller sizes and owns
 *  the memory before the step runs, so a step never fails half-done for
 *  want of it.)
 *
 * The split-KV path stores fp32 partial results (m, l, acc[D]) per
 * (query row, split, head). The bound uses host-known scalars: B lanes, T
 * rows, the largest ctx_len, and total_ctx (sum of ctx_lens over lanes; pass
 * a negative value if unknown, which gives a looser bound).
 * Returns 0 for unsupported arguments.
 */
size_t pa_attention_workspace_bytes(int32_t B, int32_t T, int32_t max_q_len,
                                    int32_t max_ctx_len, int64_t total_ctx, int32_t H,
                                    int32_t Hkv, int32_t D, int32_t block_size,
                                    pa_dtype dtype);

/*
 * pa_attention_workspace_bytes_ex -- the same for an invariance mode
 * (pa_attention_workspace_bytes is this with PA_MODE_BATCH_INVARIANT). In
 * PA_MODE_ROW_INVARIANT every row holds split partials, so the bound is
 * T * ceil(max_ctx_len / 512) (row, split) pairs. The PA_MODE_REUSE_PLAN bit
 * changes nothing here. Returns 0 for unsupported arguments or an unknown
 * mode.
 */
size_t pa_attention_workspace_bytes_ex(int32_t B, int32_t T, int32_t max_q_len,
                                       int32_t max_ctx_len, int64_t total_ctx, int32_t H,
                                       int32_t Hkv, int32_t D, int32_t block_size,
                                       pa_dtype dtype, pa_mode mode);

/*
 * pa_attention -- attention of one flat ragged step.
 * ("P3: native paged-KV continuous-batching sampler", Design, paged.py: the
 *  PagedAttention protocol -- write new K/V, return [T, H, D] -- and the
 *  paged-attention kernel contract: q, k/v cache blocks, block tables,
 *  cu_seqlens_q, ctx_lens, slot mapping; fixed KV split per context length,
 *  no atomics. Read here as: no result accumulated atomically. The kernels
 *  take their work items from atomic counters in the workspace, which
 *  decides only which warp or CTA computes an item, never its arithmetic.)
 *
 *   q                [T, H, D]
 *   k_cache, v_cache [num_blocks, block_size, Hkv, D]
 *   block_tables     int32 [B, max_blocks_per_seq]; entries past
 *                    ceil(ctx_len / block_size) are never read
 *   cu_seqlens_q     int32 [B + 1]; cu[0] = 0, cu[B] = T, non-decreasing
 *   ctx_lens         int32 [B]
 *   slot_mapping, k_new, v_new
 *                    optional (all NULL or all set): when set, the rows are
 *                    written first on the same stream, exactly as
 *                    pa_write_kv does, and attention sees them
 *   out              [T, H, D] (dtype of q); rows of lanes with q_len = 0 do
 *                    not exist; every other row is written
 *   max_q_len, max_ctx_len
 *                    host upper bounds over lanes, used only to size grids
 *   scale            softmax scale applied to q.k (fp32, finite and > 0)
 *   workspace        device scratch of workspace_bytes >= the value
 *                    pa_attention_workspace_bytes returns for this step,
 *                    256-byte aligned; contents on entry are irrelevant.
 *                    The call's kernels own it until its work on `stream`
 *                    completes (the split plan, the kernels' item counters
 *                    and the split partials live there): calls whose work
 *                    may overlap on the GPU need separate workspaces
 * Lanes with q_len == 1 take the split-KV decode path: a row with K keys is
 * split into ranges [S i, S (i + 1)) with S = 512 * 2^j for the smallest j
 * that gives at most 128 ranges (512-key ranges up to K = 65536), each range
 * reduced in ascending key order, and the ranges folded left to right in
 * fp32. In bf16 steps lanes with q_len >= 2 take the tensor-core prefill
 * path; fp32 steps take the split path for every row. Which path a row
 * takes, its split points and its reduction order depend only on its own
 * lane.
 */
pa_status pa_attention(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                       const int64_t* slot_mapping, const void* k_new, const void* v_new,
                       void* out, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t D,
                       int32_t block_size, int32_t num_blocks, int32_t max_q_len,
                       int32_t max_ctx_len, float scale, pa_dtype dtype, void* workspace,
                       size_t workspace_bytes, int32_t* status, void* stream);

/*
 * pa_attention_ex -- pa_attention with cache scales, an invariance mode and
 * phase timing hooks (pa_attention is this with scales 1,
 * PA_MODE_BATCH_INVARIANT and no events; it refuses PA_FP8_E4M3 with
 * PA_ERR_UNSUPPORTED).
 *   k_scale, v_scale
 *             scales of PA_FP8_E4M3 caches (finite and > 0, else
 *             PA_ERR_INVALID_ARG); ignored for the other types. e4m3 steps
 *             take the split path for every row (as fp32 steps do), so they
 *             are row invariant in either mode; scores use
 *             scale * k_scale and every output is multiplied by v_scale.
 *   mode      see pa_mode: an invariance mode, optionally with the
 *             PA_MODE_REUSE_PLAN bit; any other value returns
 *             PA_ERR_INVALID_ARG. The workspace must hold what
 *             pa_attention_workspace_bytes_ex returns for the same mode.
 *   events    array of n_events cudaEvent_t handles (may be NULL / 0). They
 *             are recorded on `stream` in this order, as far as n_events
 *             reaches: [0] before the first launch, [1] after the write +
 *             plan prologue, [2] after the work launch (the split kernel, or
 *             on steps with prefill rows the launch that runs the split work
 *             and the prefill side by side), [3] at the same point (the
 *             prefill has no launch of its own), [4] after the combine.
 *             When `stream` is being captured into a CUDA graph the events
 *             become event-record nodes of the graph (recorded at each
 *             replay).
 */
pa_status pa_attention_ex(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                          const int64_t* slot_mapping, const void* k_new, const void* v_new,
                          void* out, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t D,
                          int32_t block_size, int32_t num_blocks, int32_t max_q_len,
                          int32_t max_ctx_len, float scale, pa_dtype dtype, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream,
                          float k_scale, float v_scale, pa_mode mode, void* const* events,
                          int32_t n_events);

/*
 * KV-parallel page owners ("Numerics envelopes", Layout invariance of query
 * context parallelism: combine_attention_partials merges the partials of the
 * KV-parallel page owners with the ordered fold; The hierarchy: a reduction
 * is data movement plus a fixed-order fp32 fold of ranks 0..W-1).
 *
 * The keys of each lane are spread over W owners: owner w holds keys
 * [bound_w, bound_{w+1}) of lane b, with bound_0 = 0, bound_W >= ctx_len and
 * every interior bound a multiple of split_len(ctx_len) (the split length of
 * the lane's longest row; see pa_attention), so every split of every row
 * belongs to exactly one owner. Every row of the step (decode or prefill)
 * takes the split path, as in PA_MODE_ROW_INVARIANT. Each owner computes the
 * partials of its own splits into its copy of a partial buffer, the copies
 * are gathered (an all-gather: W buffers back to back), and the merge folds
 * every row's splits in global split order. The result is bitwise the
 * single-owner PA_MODE_ROW_INVARIANT result, for any W and any bounds.
 *
 * Partial buffer (pa_partials_bytes bytes, 256-byte aligned): entry
 * e(row, i) = base(row) + i for split i of flat row `row`, base(row) = the
 * number of splits of all earlier rows; an entry holds (m, l) per head
 * (float2 [H], m in the log2 domain) in the first region and acc per head
 * (float [H][D]) in the second, both sized for T * ceil(max_ctx_len / 512)
 * entries. Entries of splits another owner holds are left untouched.
 */
size_t pa_partials_bytes(int32_t T, int32_t max_ctx_len, int32_t H, int32_t D);

/* Device scratch of pa_attention_partials / pa_merge_partials (their split
 * plans); 0 for negative sizes. */
size_t pa_partials_workspace_bytes(int32_t B, int32_t T, int32_t max_ctx_len);

/*
 * pa_attention_partials -- this owner's split partials.
 *   key_lo, key_hi  int32 [B] (device): the keys [key_lo[b], key_hi[b]) of
 *                   lane b this owner holds (split-aligned as above, else
 *                   PA_FLAG_OWNER_RANGE and the lane is skipped). Only block
 *                   table entries of those keys are read.
 *   partials        this owner's partial buffer (partials_bytes >=
 *                   pa_partials_bytes(T, max_ctx_len, H, D))
 * The other arguments are pa_attention_ex's (no KV write: the owner of a new
 * row's page writes it with pa_write_kv_scaled). out is not written.
 */
pa_status pa_attention_partials(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                const int32_t* key_lo, const int32_t* key_hi, int32_t B,
                                int32_t T, int32_t H, int32_t Hkv, int32_t D,
                                int32_t block_size, int32_t num_blocks, int32_t max_q_len,
                                int32_t max_ctx_len, float scale, pa_dtype dtype, float k_scale,
                                float v_scale, void* partials, size_t partials_bytes,
                                void* workspace, size_t workspace_bytes, int32_t* status,
                                void* stream);

/*
 * pa_merge_partials -- fold the gathered partials of W owners into out.
 *   partials     W owner buffers of partials_bytes each, back to back (owner
 *                w at byte w * partials_bytes), as an all-gather leaves them
 *   key_bounds   int32 [W + 1][B] (device): row w holds bound_w of every lane
 *   v_scale      the V scale of PA_FP8_E4M3 caches (outputs are multiplied
 *                by it), ignored otherwise
 * Every row's splits are folded left to right in fp32, split i read from the
 * owner whose range holds its first key; out gets A / L (times v_scale)
 * rounded to the q dtype. Lanes with malformed bounds set
 * PA_FLAG_OWNER_RANGE and are skipped.
 */
pa_status pa_merge_partials(const void* partials, size_t partials_bytes, int32_t W,
                            const int32_t* key_bounds, const int32_t* cu_seqlens_q,
                            const int32_t* ctx_lens, void* out, int32_t B, int32_t T, int32_t H,
                            int32_t D, int32_t max_q_len, int32_t max_ctx_len, pa_dtype dtype,
                            float v_scale, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream);

/*
 * pa_decode_gemm -- batch-invariant decode linear layer at a fixed token width
 * ("ninfer" issue 80, Proposal: opt-in fixed decode width: every GEMM-class
 * decode op runs at a fixed width T_pad with padded activations, so its
 * kernel and internal schedule are the same for every real token count
 * t <= T_pad, and padding columns never mix into real ones).
 *
 *   x  [T_pad, K] bf16   rows t >= the real token count are padding (any
 *                        bits, NaN included); they only reach their own
 *                        output rows
 *   w  [N, K] bf16       the weight, row-major (y = x w^T)
 *   y  [T_pad, N] bf16   y[t, n] = sum_k x[t, k] w[n, k]: fp32 accumulation,
 *                        rounded once to bf16
 *   T_pad in {32, 64, 96, 128, 192, 256}; N a multiple of 128; K a multiple
 *   of 64 (else PA_ERR_UNSUPPORTED); pointers 16-byte aligned.
 * The schedule -- 128-row weight tiles, S splits of K whose partial sums
 * are added in split order -- is a function of (N, K) only
 * (pa_decode_gemm_splits); so y[t, :] depends on x[t, :] and w alone, never
 * on the other rows of x or on how many of them are real.
 * workspace: pa_decode_gemm_workspace_bytes(T_pad, N, K) bytes, 256-byte
 * aligned (0 bytes, and NULL allowed, when S = 1).
 */
int32_t pa_decode_gemm_splits(int32_t N, int32_t K);
size_t pa_decode_gemm_workspace_bytes(int32_t T_pad, int32_t N, int32_t K);
pa_status pa_decode_gemm(const void* x, const void* w, void* y, int32_t T_pad, int32_t N,
                         int32_t K, void* workspace, size_t workspace_bytes, int32_t* status,
                         void* stream);

/*
 * pa_attention_static_scratch -- pa_attention for callers that cannot
 * allocate device memory. (No counterpart in the paper: this entry point
 * exists for integration, not for the method.)
 *
 * Some callers cannot call cudaMalloc where they run a step: a plugin whose
 * host framework offers it no device allocator, a process whose memory pool
 * has claimed all free device memory up front, or a latency-critical loop
 * that cannot take the device-wide synchronisation cudaMalloc / cudaFree may
 * cause. This entry point takes the same inputs and outputs as pa_attention
 * but no workspace: its split-KV scratch is one array of
 * PA_STATIC_SCRATCH_BYTES compiled into the library. It calls no cudaMalloc,
 * cudaFree or other allocating routine (see Set-up for when the array's own
 * memory is taken).
 *
 *   total_ctx  sum of ctx_lens over the lanes (negative if unknown), used
 *              with B, T, max_q_len and max_ctx_len to bound the scratch the
 *              step needs, exactly as pa_attention_workspace_bytes does.
 * Returns PA_ERR_INVALID_ARG for negative sizes (as pa_attention does) and
 * PA_ERR_WORKSPACE when that bound exceeds PA_STATIC_SCRATCH_BYTES, both
 * before any CUDA call; PA_ERR_UNSUPPORTED for unsupported geometry.
 * Set-up: the first call on each device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress) and keeps it. That
 * lookup is also when CUDA loads the library part holding the array and
 * takes its PA_STATIC_SCRATCH_BYTES of device memory (lazy module loading,
 * CUDA's default): a caller whose memory pool will claim all free device
 * memory, or that captures streams into graphs, makes one set-up call first
 * -- a call with B = T = 0 (any supported geometry, num_blocks >= 1, a
 * positive scale) does only the set-up and returns PA_OK. From then on the device holds the array until the process exits,
 * and calls allocate nothing. The kept address belongs to the device's
 * context at set-up: do not call again after a cudaDeviceReset of that
 * device. Every call on a device shares the one array and it keeps the last
 * call's contents (nothing in it needs to start at zero: each call rewrites
 * the plan and partials it reads); calls whose work overlaps on the GPU --
 * on different streams, or from different threads -- race on it and must be
 * serialised by the caller.
 */
#define PA_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

pa_status pa_attention_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                      const int64_t* slot_mapping, const void* k_new,
                                      const void* v_new, void* out, int32_t B, int32_t T,
                                      int32_t H, int32_t Hkv, int32_t D, int32_t block_size,
                                      int32_t num_blocks, int32_t max_q_len, int32_t max_ctx_len,
                                      int64_t total_ctx, float scale, pa_dtype dtype,
                                      int32_t* status, void* stream);

/*
 * pa_read_status -- wait for `stream`, copy the device status word to
 * *flags_out and, if clear != 0, reset it to zero. The only synchronising call.
 * ("P3: native paged-KV continuous-batching sampler", Review (adversarial
 *  pass): an out-of-vocabulary prompt id became a device-side assert that
 *  wedged the engine, and greedy NaN logits passed silently; both now fail
 *  loudly before any sequence advances. Read here as: a bad index seen only
 *  on the device never traps a kernel -- it sets a PA_FLAG_* bit that the
 *  caller reads here, after the step, and acts on.)
 */
pa_status pa_read_status(int32_t* status, void* stream, int32_t* flags_out, int32_t clear);

/* Human-readable name of a pa_status value (static storage).
 * (Host-visible refusals are returned at entry, before any launch: "P3:
 *  native paged-KV continuous-batching sampler", Review (adversarial pass),
 *  bad requests refused at add_request instead of wedging the engine;
 *  "Numerics envelopes", Precedence: refuse a choice that would void the
 *  contract rather than keep it silently.) */
const char* pa_status_string(pa_status s);

/* Kernels this process has launched through the library so far. */
int64_t pa_kernel_launches(void);

/* Shortest split length (keys) of the decode path; longer rows use the
 * power-of-two multiple of it that keeps them at most 128 splits. */
int32_t pa_split_tokens(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
