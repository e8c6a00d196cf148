/*
 * mha.h - C ABI of the GB300 multi-head attention forward pass.
 *
 * The layer (the "Multi-head attention and self-attention" Definition on
 * alphabetamath.cc, and the "The Complete Multi-Head Operation" section of
 * the llmprimer.com multi-head attention review):
 *
 *   head i:  H_i = softmax( c * (X_q W_i^Q)(X_kv W_i^K)^T + M ) (X_kv W_i^V)
 *   output:  Y   = Concat_feature(H_1, ..., H_h) W^O
 *
 * computed on one GPU in three steps, each also exported on its own:
 *   1. mha_qkv_projection   - combined projections with the head split
 *                             (B,T,h*d) -> (B,h,T,d) done in the GEMM epilogue;
 *   2. mha_attention        - the fused attention kernel: key blocks are folded
 *                             into the stable summary (m, l, z) with its merge
 *                             ("Stable summary of an attention key block",
 *                             Definition), z / l is taken once per row, and the
 *                             B x h x n_q x n_k score tensor is never stored;
 *   3. mha_output_projection - Y = Z W^O.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensors are dense, row-major, batch-major ("The Complete Multi-Head
 *   Operation": X : B x T x d_model, Z : B x T x (h d_v), Y : B x T x d_model).
 * - Weights are used as given, right-multiplied (X W), in the combined form of
 *   "Separate and Combined Projections": W_Q, W_K are d_model x (h*d_h) and
 *   W_V is d_model x (h*d_vh); head i owns columns [i*d, (i+1)*d). W_O is
 *   (h*d_vh) x d_o; head i owns rows [i*d_vh, (i+1)*d_vh). No biases.
 * - Element type: MHA_DTYPE_BF16 (inputs, intermediates and Y in bf16,
 *   accumulation in fp32, tensor cores) or MHA_DTYPE_F32 (everything fp32,
 *   CUDA-core FMA kernels).
 * - Pointers named X_*, W_*, Q, K, V, Z, Y and the workspace are DEVICE
 *   pointers owned by the caller; the library keeps none of them after the
 *   call returns and allocates no device memory. `valid_len` is a HOST array.
 *   Every device pointer must be 16-byte aligned. Outputs must not alias
 *   inputs; X_kv may equal X_q.
 * - `stream` is a cudaStream_t (NULL = legacy default stream). Every call is
 *   asynchronous on that stream: it validates its arguments on the host,
 *   enqueues its kernels and returns.
 * - Masks ("From Attention to Self-Attention review", "Causal and padding
 *   masks"; masked positions get weight exactly 0):
 *     MHA_MASK_NONE            every query row uses every key;
 *     MHA_MASK_CAUSAL          row i uses keys j <= i (needs n_q == n_k);
 *     MHA_MASK_PADDING         batch item b uses keys j < valid_len[b];
 *     MHA_MASK_CAUSAL_PADDING  both.
 *   In self-attention (X_kv == NULL) with a padding mask the query rows
 *   i >= valid_len[b] are padding as well: they are not computed and their
 *   rows of Z and Y are written as exact zeros. In cross-attention the
 *   padding applies to keys only.
 * - Every query row must keep at least one allowed key (the nonempty allowed
 *   set of the block-summary Definition): valid_len[b] must lie in
 *   [1, n_k], else the call returns MHA_ERR_EMPTY_ROW and launches nothing.
 *
 * Errors: arguments are checked on the host before anything is enqueued; on
 * any error nothing is launched and the outputs are untouched. A kernel that
 * waits too long on one of its own barriers gives up, records
 * MHA_ERR_DEVICE_TIMEOUT in the caller's device error word and returns; read it
 * with mha_get_device_error.
 */
#ifndef MHA_GB300_H
#define MHA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MHA_API __attribute__((visibility("default")))
#else
#define MHA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MHA_OK = 0,
  MHA_ERR_INVALID_ARG = 1,    /* a NULL or non-positive argument, a bad enum, non-finite c */
  MHA_ERR_UNSUPPORTED = 2,    /* a valid shape the library does not handle (see mha_forward) */
  MHA_ERR_EMPTY_ROW = 3,      /* some query row would have no allowed key */
  MHA_ERR_WORKSPACE = 4,      /* workspace NULL, misaligned or smaller than mha_workspace_size */
  MHA_ERR_CUDA = 5,           /* a CUDA runtime call or a launch failed */
  MHA_ERR_DEVICE_TIMEOUT = 6  /* a kernel gave up waiting on one of its barriers */
} mha_status;

typedef enum {
  MHA_MASK_NONE = 0,
  MHA_MASK_CAUSAL = 1,
  MHA_MASK_PADDING = 2,
  MHA_MASK_CAUSAL_PADDING = 3
} mha_mask_kind;

typedef enum { MHA_DTYPE_F32 = 0, MHA_DTYPE_BF16 = 1 } mha_dtype;

/* Largest batch accepted together with a padding mask (the valid lengths
 * travel to the kernels inside their launch parameters). */
#define MHA_MAX_PADDED_BATCH 1024

/* Most heads a head gate (mha_forward_general) may address. */
#define MHA_MAX_GATED_HEADS 1024

/* Largest split over the keys mha_attention_split and mha_attention_plan take. */
#define MHA_MAX_KEY_SPLITS 256

/*
 * Bytes of device workspace mha_forward needs for these sizes: the head-split
 * Q, K (B*h*n*d_h elements), V (B*h*n_k*d_vh), the concatenated Z
 * (B*n_q*h*d_vh), a 256-byte header whose first int32 is the device error
 * word, and, for bf16 heads on the tensor cores with few query tiles, the
 * scratch of the automatic split over the keys (see mha_attention_split:
 * mha_attention_split_workspace_size with nsplit = 0, at most about 21 MB).
 * Linear in n_q and n_k: no term grows with n_q * n_k. Returns 0 when an
 * argument is non-positive or the dtype is unknown.
 */
MHA_API size_t mha_workspace_size(int B, int n_q, int n_k, int d_model, int h, int d_h,
                          int d_vh, int d_o, mha_dtype dt);

/*
 * Byte offsets inside the workspace of mha_forward, for callers that want to
 * inspect the intermediates or run the three steps themselves on the same
 * buffers: offsets[0] the int32 device error word, [1] Q, [2] K, [3] V, [4] Z,
 * [5] the total size (= mha_workspace_size). The bytes between the end of Z
 * (rounded up to 1 KB) and the total are the split scratch. Returns
 * MHA_ERR_INVALID_ARG on a non-positive size, an unknown dtype or a NULL
 * `offsets`.
 */
MHA_API mha_status mha_workspace_layout(int B, int n_q, int n_k, int h, int d_h, int d_vh,
                                        mha_dtype dt, size_t offsets[6]);

/*
 * The whole forward pass: Y = MHA(X_q, X_kv).
 *
 *   X_q   (B, n_q, d_model)      queries' token matrix
 *   X_kv  (B, n_k, d_model)      keys' and values' token matrix; NULL means
 *                                self-attention (X_kv := X_q, needs n_k == n_q)
 *   W_Q, W_K (d_model, h*d_h), W_V (d_model, h*d_vh), W_O (h*d_vh, d_o)
 *   Y     (B, n_q, d_o)          output
 *   c                            score scale (finite; 1/sqrt(d_h) is usual)
 *   valid_len                    HOST int32[B] for the padding masks, else
 *                                ignored (may be NULL)
 *   workspace, workspace_bytes   device scratch of at least
 *                                mha_workspace_size(...) bytes, 256-byte
 *                                aligned; its contents on entry do not matter
 *
 * Head sizes d_h, d_vh from 1 to 256 (MHA_ERR_UNSUPPORTED otherwise); bf16
 * heads with d_h and d_vh in 32..128 and multiples of 8 run on the tensor
 * cores (sizes of 32..64 in the 64-wide kernels, sizes above 64 in the
 * 128-wide ones, the columns past d_h or d_vh read as zeros), other sizes on
 * CUDA cores.
 * bf16 also needs d_model, d_h, d_vh and d_o to be multiples of 8.
 * When the bf16 tile pairs of the attention step are too few to fill the
 * GPU, the step splits the keys as mha_attention_split does with nsplit = 0,
 * in the workspace's split scratch (one more small memset, of its counters).
 * Enqueues a 4-byte memset of the error word and three kernels. Everything
 * it enqueues is stream-ordered, so the call can be captured in a CUDA graph
 * on fixed buffers and replayed; host-side arguments (sizes, c, valid_len)
 * are read at capture time and stay fixed in the replays.
 */
MHA_API mha_status mha_forward(const void* X_q, const void* X_kv, const void* W_Q,
                       const void* W_K, const void* W_V, const void* W_O,
                       void* Y, int B, int n_q, int n_k, int d_model, int h,
                       int d_h, int d_vh, int d_o, float c, mha_mask_kind mask,
                       const int32_t* valid_len, mha_dtype dt, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * The forward pass in the general form of "Multi-head attention and
 * self-attention" (alphabetamath.cc, Definition): query, key and value
 * inputs are three matrices of their own widths,
 *   head i = Attn(X_q W_i^Q, X_k W_i^K, X_v W_i^V),  Y = Concat(heads) W^O.
 *
 *   X_q (B, n_q, d_q), X_k (B, n_k, d_k), X_v (B, n_k, d_v); X_k and X_v may
 *                                be the same buffer, and so may X_q (self-
 *                                attention passes X_q three times)
 *   W_Q (d_q, h*d_h), W_K (d_k, h*d_h), W_V (d_v, h*d_vh), W_O (h*d_vh, d_o)
 *   Y (B, n_q, d_o)
 *   self_attention != 0          rows i >= valid_len[b] are padding queries
 *                                (not computed, Y rows 0); needs n_q == n_k.
 *                                0: a padding mask applies to keys only
 *   head_gate                    HOST float[h] or NULL: head i's output block
 *                                of the concatenation (columns [i*d_vh,
 *                                (i+1)*d_vh) of Z, before W^O) is multiplied
 *                                by head_gate[i]; 0 ablates the head, which
 *                                equals zeroing row block i of W^O ("Head
 *                                Identity and Ablation", Multi-Head Attention
 *                                review). NULL: every gate is 1. With a gate,
 *                                h <= MHA_MAX_GATED_HEADS (else
 *                                MHA_ERR_UNSUPPORTED); gates must be finite
 *                                (else MHA_ERR_INVALID_ARG)
 *   workspace                    as for mha_forward (mha_workspace_size with
 *                                any d_model: the intermediates do not depend
 *                                on the input widths)
 *
 * Head sizes d_h, d_vh from 1 to 256; bf16 heads with d_h and d_vh in 32..128
 * (multiples of 8) run on the tensor cores (as for mha_forward), other sizes
 * on CUDA cores.
 * bf16 also needs d_q, d_k, d_v,
 * d_h, d_vh and d_o to be multiples of 8 and 16-byte aligned pointers
 * (MHA_ERR_UNSUPPORTED otherwise). Other errors as for mha_forward.
 * mha_forward is this call with X_k = X_v = X_kv (or X_q) and
 * d_q = d_k = d_v = d_model.
 */
MHA_API mha_status mha_forward_general(const void* X_q, const void* X_k, const void* X_v,
                                       const void* W_Q, const void* W_K, const void* W_V,
                                       const void* W_O, void* Y, int B, int n_q, int n_k,
                                       int d_q, int d_k, int d_v, int h, int d_h, int d_vh,
                                       int d_o, float c, mha_mask_kind mask,
                                       const int32_t* valid_len, int self_attention,
                                       const float* head_gate, mha_dtype dt, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * Step 1: combined projections with the head split ("Separate and Combined
 * Projections": (B,T,h d) -> (B,T,h,d) -> (B,h,T,d)).
 *   Q (B, h, n_q, d_h) = head split of X_q W_Q
 *   K (B, h, n_k, d_h) = head split of X_kv W_K
 *   V (B, h, n_k, d_vh) = head split of X_kv W_V
 * X_kv NULL means X_kv := X_q (n_k must equal n_q). dev_error: device int32
 * error word (may be NULL: timeouts then go unreported).
 * mask, valid_len: as for mha_attention. With a padding mask (bf16) only the
 * rows mha_attention reads are computed: rows j < valid_len[b] rounded up to
 * a multiple of 128 (capped at n_k) of K and V, and the same rows of Q for
 * self-attention (X_kv NULL); the rows past them are left as they were. The
 * rows between valid_len[b] and that bound are computed because mha_attention
 * reads them (with weight exactly 0, so they must be finite).
 * MHA_ERR_INVALID_ARG for a padding mask without valid_len, MHA_ERR_EMPTY_ROW
 * for a length outside [1, n_k].
 */
MHA_API mha_status mha_qkv_projection(const void* X_q, const void* X_kv,
                              const void* W_Q, const void* W_K, const void* W_V,
                              void* Q, void* K, void* V, int B, int n_q,
                              int n_k, int d_model, int h, int d_h, int d_vh,
                              mha_mask_kind mask, const int32_t* valid_len,
                              mha_dtype dt, int32_t* dev_error, void* stream);

/*
 * Step 2: fused masked attention on head-split inputs, written in the
 * concatenated layout ("reverse the head-position transpose", then
 * "Concatenate along the head-feature axis in the declared order").
 *   Q (B, h, n_q, d_h), K (B, h, n_k, d_h), V (B, h, n_k, d_vh)
 *   Z (B, n_q, h*d_vh): Z[b, i, j*d_vh + r] = head j's output row i, column r
 * self_attention != 0 marks the padded query rows (i >= valid_len[b]) as not
 * computed (their Z rows are 0); 0 applies padding to keys only.
 */
MHA_API mha_status mha_attention(const void* Q, const void* K, const void* V, void* Z,
                         int B, int n_q, int n_k, int h, int d_h, int d_vh,
                         float c, mha_mask_kind mask, const int32_t* valid_len,
                         int self_attention, mha_dtype dt, int32_t* dev_error,
                         void* stream);

/*
 * Bytes of device scratch mha_attention_split needs: nsplit = 0 (the
 * automatic choice) the most it may use for these sizes, 0 when it would
 * never split; nsplit >= 1 that split (0 for nsplit = 1, or when n_k has a
 * single 128-key block). The scratch holds one int counter per query tile,
 * then one summary per (query tile, key range): z (d_vh rounded up to 64 or
 * 128 columns), m and l of its 128 rows, in fp32. 0 for non-positive sizes
 * or head sizes outside the tensor-core path.
 */
MHA_API size_t mha_attention_split_workspace_size(int B, int n_q, int n_k, int h, int d_h,
                                                  int d_vh, int nsplit);

/*
 * Step 2 with the keys of each (query tile, head) cut into ranges that run on
 * separate thread blocks ("Stable summary of an attention key block",
 * alphabetamath.cc, Definition: the summary of a union of disjoint key sets
 * is the merge of their summaries). For few query rows over many keys, such
 * as a short query block against a long key sequence, the tile pairs alone
 * would leave most SMs idle. Each range folds its key blocks into its own
 * summary (m, l, z) of every row and publishes it in the scratch; the thread
 * block that publishes the last range of a tile merges the tile's summaries
 * in range order (m' = max m_s, l' = sum e^{m_s - m'} l_s, z' likewise) and
 * writes z' / l' to Z. No thread block waits for another.
 *   nsplit      0: automatic (a split only when the tile pairs leave SMs
 *               idle and the estimate is shorter, within workspace_bytes);
 *               1: none (as mha_attention); n in 2..MHA_MAX_KEY_SPLITS: the
 *               128-key blocks of n_k cut into n ranges of equal whole blocks
 *               (fewer ranges when they do not divide); any mask. A range
 *               that holds no allowed key of a tile (past a valid length,
 *               past the causal diagonal) is the empty summary.
 *   workspace   device scratch of mha_attention_split_workspace_size bytes,
 *               256-byte aligned, contents on entry irrelevant (its counters
 *               are zeroed by a memset this call enqueues); may be NULL for
 *               nsplit 0 or 1
 * Other arguments as for mha_attention. Errors as for mha_attention, and:
 * MHA_ERR_INVALID_ARG for nsplit outside [0, MHA_MAX_KEY_SPLITS];
 * MHA_ERR_UNSUPPORTED for nsplit > 1 with fp32 or head sizes off the tensor
 * cores; MHA_ERR_WORKSPACE for a missing, misaligned or small workspace.
 * Calls sharing a workspace must not overlap on the GPU.
 */
MHA_API mha_status mha_attention_split(const void* Q, const void* K, const void* V, void* Z,
                                       int B, int n_q, int n_k, int h, int d_h, int d_vh,
                                       float c, mha_mask_kind mask, const int32_t* valid_len,
                                       int self_attention, int nsplit, mha_dtype dt,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* dev_error, void* stream);

/*
 * The schedule of the tensor-core attention for bf16 heads (d_h and d_vh in
 * 32..128, multiples of 8), computed on the host for a GPU with num_sms SMs;
 * it launches nothing and needs no GPU. nsplit as for mha_attention_split:
 * 1 is the schedule of mha_attention, 0 that of mha_forward (the automatic
 * split with the scratch mha_workspace_size provides). A unit is one 128-row
 * query tile or a pair of them, of one (batch item, head), over a range of
 * keys; each CTA of the grid takes its units in order. Outputs:
 *   *grid        CTAs the launch would use (num_sms for the persistent
 *                schedule, the number of units for one CTA per unit)
 *   records      HOST int32 array of 7 * max_records (may be NULL): for each
 *                unit, CTA by CTA in processing order, {cta, b, head, q0,
 *                ntiles, key0, key1}: query rows [q0, q0 + 128 ntiles) of
 *                head `head` of batch item b (rows at or past n_q do not
 *                exist) over keys [key0, key1) (before the mask); at most
 *                max_records records are written
 *   *n_records   the number of units (records needed)
 * Arguments as for mha_attention; MHA_ERR_INVALID_ARG on a NULL grid or
 * n_records, num_sms < 1, nsplit outside [0, MHA_MAX_KEY_SPLITS] or an
 * invalid size or mask, MHA_ERR_EMPTY_ROW on a bad valid length,
 * MHA_ERR_UNSUPPORTED for other head sizes.
 */
MHA_API mha_status mha_attention_plan(int B, int n_q, int n_k, int h, int d_h, int d_vh,
                              mha_mask_kind mask, const int32_t* valid_len,
                              int self_attention, int nsplit, int num_sms, int32_t* grid,
                              int32_t* records, size_t max_records, size_t* n_records);

/*
 * Step 3: Y (B*n_q, d_o) = Z (B*n_q, h*d_vh) W_O (h*d_vh, d_o)
 * ("The Complete Multi-Head Operation": Y = Z W_O).
 * valid_len: HOST int32[B] or NULL. Given, the rows i >= valid_len[b] of
 * batch item b are the padded query rows of self-attention, whose Z rows
 * mha_attention writes as zeros: Y there is zero, and (bf16) 128-row panels
 * made only of such rows are written as zeros without a product.
 * MHA_ERR_EMPTY_ROW for a length outside [1, n_q].
 */
MHA_API mha_status mha_output_projection(const void* Z, const void* W_O, void* Y,
                                 int B, int n_q, int h, int d_vh, int d_o,
                                 const int32_t* valid_len, mha_dtype dt,
                                 int32_t* dev_error, void* stream);

/*
 * Device scratch for mha_attention_decode, in bytes: one partial summary
 * (m, l and d_vh values of z, fp32) per query row, head, batch item and
 * split of the cache (one per 128 cache positions); 0 when an argument is
 * non-positive.
 */
MHA_API size_t mha_decode_workspace_size(int B, int n_q, int n_k, int h, int d_vh);

/*
 * Attention of a few new query rows over a key/value cache: the workload of
 * autoregressive generation named in "From Attention to Self-Attention
 * review" (each new token attends to the cached positions), computed with the
 * summary and merge of "Stable summary of an attention key block"
 * (alphabetamath.cc, Definition): the cache is cut into splits, each split is
 * summarised on its own, and the summaries are merged.
 *
 *   Q (B, h, n_q, d_h)    the new rows, head-split
 *   K (B, h, n_k, d_h)    the cache, capacity n_k; batch item b holds
 *   V (B, h, n_k, d_vh)   cache_len[b] valid positions 0 .. cache_len[b]-1
 *   Z (B, n_q, h*d_vh)    output, concatenated layout (as mha_attention)
 *   cache_len             HOST int32[B], each in [1, n_k]; NULL: all n_k
 *   causal_tail           0: every row sees all cache_len[b] keys. 1: the n_q
 *                         rows are the last positions of the sequence and row i
 *                         sees keys j <= cache_len[b] - n_q + i (needs
 *                         cache_len[b] >= n_q)
 *   workspace             device scratch of mha_decode_workspace_size bytes,
 *                         16-byte aligned, contents on entry irrelevant
 *
 * Errors (host checks before any launch): MHA_ERR_INVALID_ARG for NULL
 * pointers, non-positive sizes, non-finite c; MHA_ERR_EMPTY_ROW for a cache
 * length outside [1, n_k] (or below n_q with causal_tail);
 * MHA_ERR_UNSUPPORTED for B above MHA_MAX_PADDED_BATCH, d_h or d_vh above
 * 256, n_k above 65536, bf16 with d_h not a multiple of 8 or misaligned
 * pointers; MHA_ERR_WORKSPACE for a missing or small workspace. Enqueues two
 * kernels; asynchronous.
 */
MHA_API mha_status mha_attention_decode(const void* Q, const void* K, const void* V, void* Z,
                                        int B, int n_q, int n_k, int h, int d_h, int d_vh,
                                        float c, const int32_t* cache_len, int causal_tail,
                                        mha_dtype dt, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* Size of the device scratch built into the library for mha_forward_no_alloc. */
#define MHA_NO_ALLOC_SCRATCH_BYTES (32u << 20)

/*
 * mha_forward without a workspace, for callers that cannot allocate device
 * memory: code running where cudaMalloc is forbidden or unavailable, such as
 * inside a host framework that owns every device allocation, a plugin held
 * to a fixed memory budget, or a loop that must not allocate once running.
 * The caller passes its inputs and outputs exactly as for mha_forward; the
 * intermediates (head-split Q, K, V, the concatenated Z and the device error
 * word) live in a static device array of MHA_NO_ALLOC_SCRATCH_BYTES (32 MiB)
 * that is part of the library. The pages define no such entry point: it has
 * no counterpart there.
 *
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   Every GPU on which the library's device code is loaded holds the 32 MiB
 *   until the process exits.
 * - Sizes whose intermediates need more than MHA_NO_ALLOC_SCRATCH_BYTES
 *   (mha_workspace_size(...) > 32 MiB) return MHA_ERR_WORKSPACE before any
 *   CUDA call. Other arguments are checked as in mha_forward.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, and caches it; make that
 *   first call before any stream capture on that device.
 * - Every call shares the one array and leaves its contents behind; the error
 *   word is reset at the start of each call. Calls whose work overlaps on the
 *   GPU (different streams, or other host threads) race on the array: order
 *   them on one stream or synchronise between them.
 * - A kernel that gives up on a barrier records the timeout in the array's
 *   error word, which this entry point does not read back; a caller that needs
 *   that report uses mha_forward and mha_get_device_error.
 */
MHA_API mha_status mha_forward_no_alloc(const void* X_q, const void* X_kv, const void* W_Q,
                                        const void* W_K, const void* W_V, const void* W_O,
                                        void* Y, int B, int n_q, int n_k, int d_model, int h,
                                        int d_h, int d_vh, int d_o, float c,
                                        mha_mask_kind mask, const int32_t* valid_len,
                                        mha_dtype dt, void* stream);

/*
 * Reads the device error word (the workspace base for mha_forward, or the
 * dev_error given to a step), waits for `stream`, resets the word to 0 and
 * returns what it held (MHA_OK when no kernel reported a problem), or
 * MHA_ERR_CUDA if the copy itself failed.
 */
MHA_API mha_status mha_get_device_error(void* error_word, void* stream);

/* A fixed English description of a status code. Never NULL. */
MHA_API const char* mha_status_string(mha_status s);

/*
 * Failure-detection self-test: launches one CTA whose thread waits on a
 * barrier that nothing completes, through the same bounded wait the kernels
 * use, with a limit of `limit_ns` nanoseconds (clamped to [1e3, 1e10]). The
 * kernel must give up, write MHA_ERR_DEVICE_TIMEOUT to *dev_error and return,
 * leaving the context usable.
 */
MHA_API mha_status mha_selftest_wait_timeout(int32_t* dev_error, uint64_t limit_ns,
                                     void* stream);

/* Number of kernels this library has enqueued since it was loaded. */
MHA_API uint64_t mha_kernel_launch_count(void);

/* Library version string. */
MHA_API const char* mha_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MHA_GB300_H */
