/*
 * dsa.h - C ABI of libdsa.so: the DeepSeek Sparse Attention (DSA) layer hot
 * path on one NVIDIA GB300 (sm_103a).
 *
 * The path has three stages ("DeepSeek3.2: Onboard sparse attention",
 * Background): a lightning indexer that scores every causal (query, key)
 * pair, a per-query top-k that turns the scores into an index set, and
 * attention restricted to that set, forward and backward ("Support Ring
 * Attention with DeepSeek DSA Sparse Indexer", Forward Flow / Backward Flow).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers are DEVICE pointers owned by the caller, 16-byte aligned,
 *    to contiguous row-major tensors of the shapes given below. The library
 *    never allocates or frees device memory.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call
 *    only enqueues work on it and returns; nothing synchronises except
 *    dsa_get_last_device_error().
 *  - Every call returns a dsa_status. Arguments are validated on the host
 *    before anything is launched; an unsupported shape returns
 *    DSA_ERR_UNSUPPORTED and nothing runs (there is no fallback path).
 *  - Faults found on the device (an index outside [-1, S), a bounded wait that
 *    ran out) do not trap: the kernel records a code in a device error word,
 *    skips the bad access and finishes. Read it with
 *    dsa_get_last_device_error().
 *  - "Valid" pairs: key s is valid for query t when s <= t (the causal mask
 *    q_pos >= kv_pos, diagonal included; "Support Ring Attention with
 *    DeepSeek DSA Sparse Indexer", Forward Flow step 3) and, when segment ids
 *    are given, seg[b,s] == seg[b,t] (packed documents; same page, Tests:
 *    indexer mask with segment ids).
 *  - bf16 arguments are IEEE bfloat16 bit patterns; results are rounded to
 *    nearest even from fp32.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
  DSA_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels implement */
  DSA_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than required */
  DSA_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed */
  DSA_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out */
  DSA_ERR_DEVICE = 6       /* the device reported bad input (see the code) */
} dsa_status;

typedef enum { DSA_BF16 = 0, DSA_F32 = 1 } dsa_dtype;

/* Device error codes returned by dsa_get_last_device_error(). 0 = none. The
 * low byte is the kind, the next byte the stage that reported it. */
#define DSA_DEVERR_TIMEOUT 0x01   /* a bounded mbarrier wait ran out */
#define DSA_DEVERR_BAD_INDEX 0x02 /* an index outside [-1, S) was skipped */
#define DSA_DEVERR_MISALIGNED 0x03 /* shared memory not aligned as the kernel needs */
#define DSA_STAGE_INDEXER 0x100
#define DSA_STAGE_TOPK 0x200
#define DSA_STAGE_FWD 0x300
#define DSA_STAGE_BWD 0x400
#define DSA_STAGE_LOSS 0x500
#define DSA_STAGE_LOSS_BWD 0x600

/* Human-readable name of a status. Never NULL. */
const char* dsa_status_string(int status);

/* Library version, e.g. 100 for 0.1.0. */
int dsa_version(void);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device. *code receives the first code recorded since the last read
 * (0 if none). Returns DSA_OK, or DSA_ERR_CUDA if the synchronisation failed.
 */
int dsa_get_last_device_error(void* stream, int32_t* code);

/*
 * dsa_index_scores - lightning-indexer scores.
 *
 * Defines ("DeepSeek3.2: Onboard sparse attention", Background: a per-head
 * q.k product gives the index score; "Implement QK attention head chunking
 * for CSA", Description: per-head products reduced over heads):
 *
 *     I[b,t,s] = sum_h w[b,t,h] * max(0, sum_d q_idx[b,t,h,d] * k_idx[b,s,d])
 *
 * for valid (t, s); -inf where s <= t but the document differs. Entries with
 * s > t are not written. Per-head products are never stored.
 *
 *   q_idx   bf16 [B, S, Hi, Di]
 *   k_idx   bf16 [B, S, Di]
 *   w       [B, S, Hi], fp32 (w_dtype = DSA_F32) or bf16 (DSA_BF16)
 *   seg     int32 [B, S] or NULL (NULL: one document per row)
 *   scores  fp32 [B, S, ld_scores], ld_scores >= S and a multiple of 4
 *
 * Supported: Hi in {1, 2, 4, ..., 128}, Di in {32, 64, 128}. Accumulation is
 * fp32 on the tensor cores; with inputs whose partial sums are all exact in
 * fp32 (e.g. small dyadic values) the result is exact.
 */
int dsa_index_scores(const void* q_idx, const void* k_idx, const void* w, int w_dtype,
                     const int32_t* seg, int B, int S, int Hi, int Di, float* scores,
                     int64_t ld_scores, void* stream);

/*
 * dsa_index_scores_fp8 - the same scores from 8-bit float inputs. The pages
 * note that the original indexer is an fp8 kernel over quantized activations
 * ("DeepSeek3.2: Onboard sparse attention", What this PR does, item 4). With a
 * positive scale c_s per key (k = c_s * k8):
 *
 *     I[b,t,s] = c_s * sum_h w[b,t,h] * max(0, sum_d q8[b,t,h,d] * k8[b,s,d])
 *
 * which equals the bf16 definition on the dequantized k, because ReLU is
 * positively homogeneous. A per-(query, head) scale of q belongs in w.
 *
 *   q_idx    e4m3 bytes [B, S, Hi, Di] (OCP FP8 E4M3: bias 7, no infinities)
 *   k_idx    e4m3 bytes [B, S, Di]
 *   k_scale  fp32 [B, S], every entry > 0, or NULL (all 1)
 *   w, seg, scores, ld_scores, stream: as for dsa_index_scores
 *
 * Supported: Hi in {1, 2, 4, ..., 128}, Di in {32, 64, 128}. The products run at
 * twice the bf16 tensor rate and accumulate in fp32; the scale is one fp32
 * multiply of the reduced score. Inputs that are small dyadic values (exact in
 * e4m3) with power-of-two scales give exact results, identical to
 * dsa_index_scores on the same values.
 */
int dsa_index_scores_fp8(const void* q_idx, const void* k_idx, const float* k_scale,
                         const void* w, int w_dtype, const int32_t* seg, int B, int S, int Hi,
                         int Di, float* scores, int64_t ld_scores, void* stream);

/*
 * dsa_topk - per-query top-k of the index scores ("DeepSeek3.2: Onboard
 * sparse attention", Background: non-parametric top-k token selection).
 *
 * For each (b, t) select m(t) = min(k, n(t)) valid keys (n(t) = number of
 * valid keys) with the largest score. Equal scores go to the lower key index;
 * -0.0 equals +0.0. Scores must not be NaN.
 *
 *   scores  fp32 [B, S, ld_scores]; only valid entries (s <= t) are read
 *   seg     int32 [B, S] or NULL
 *   idx     int32 [B, S, k] out: the selected keys in ascending order,
 *           slots m(t)..k-1 set to -1
 *   count   int32 [B, S] out, or NULL: m(t)
 *   vals    fp32 [B, S, k] out, or NULL: the score of the key in each slot of idx,
 *           -inf at slots holding -1. It is read back from the score row just after
 *           the row's selection (while the row is in L2), so that a consumer of the
 *           selected scores (dsa_indexer_loss with ld_scores = 0) reads k contiguous
 *           floats per row instead of gathering them from the row.
 *   ws      workspace of dsa_topk_workspace_size() bytes (may be NULL if 0)
 */
size_t dsa_topk_workspace_size(int B, int S, int k);
int dsa_topk(const float* scores, int64_t ld_scores, const int32_t* seg, int B, int S, int k,
             int32_t* idx, int32_t* count, float* vals, void* ws, size_t ws_bytes,
             void* stream);

/*
 * dsa_sparse_attn_fwd - attention over the selected keys ("Support Ring
 * Attention with DeepSeek DSA Sparse Indexer", Forward Flow step 5):
 *
 *     l_j = scale * Q[b,t,h] . K[b,s_j]      for the listed s_j with s_j <= t
 *     O[b,t,h] = sum_j softmax(l)_j V[b,s_j],   lse[b,t,h] = log sum_j exp(l_j)
 *
 * The selected set of query t is shared by all H heads. Entries of idx equal
 * to -1 and entries above the diagonal are ignored; a row with no key gets
 * O = 0 and lse = -inf. The entries of a row must be distinct.
 *
 *   Q    bf16 [B, S, H, Dqk]     K  bf16 [B, S, Hkv, Dqk]    V  bf16 [B, S, Hkv, Dv]
 *   idx  int32 [B, S, k]         O  bf16 [B, S, H, Dv] out   lse fp32 [B, S, H] out
 *
 * Supported: 1 <= H <= 128 and
 *  - Hkv = 1 (one K/V row shared by every head, the form the indexer's
 *    selection is built for): (Dqk, Dv) in {(32, 32), (64, 64), (128, 128),
 *    (192, 128)};
 *  - Hkv > 1 dividing H (per-head K/V, Hkv = H, or groups of H / Hkv heads;
 *    head h reads K/V head h / (H / Hkv)): the dense-tile kernel only, so
 *    (Dqk, Dv) in {(128, 128), (192, 128)}, S <= 65536 and a positive scale;
 *    DSA_ERR_UNSUPPORTED otherwise.
 *
 * Two tensor-core kernels compute it. One gathers each query's selected K/V
 * rows and puts the heads on the 128 lanes of a tile. The other evaluates dense
 * 128 x 128 (query, key) tiles of one head under a bitmap of the selection and
 * skips tiles without a selected key (see dsa_sparse_attn_fwd_dense). The call
 * takes the one with fewer tile products for the shape.
 *
 *   ws  workspace of dsa_sparse_attn_fwd_workspace_size() bytes, 16-byte aligned:
 *       the dense-tile kernel's selection bitmap and tile flags (overwritten). It
 *       is reserved whenever that kernel can take the shape, whichever kernel
 *       the call then picks; where the size is 0, ws may be NULL.
 *
 * DSA_ERR_WORKSPACE if ws is NULL, misaligned or smaller than the size (when the
 * size is not 0).
 */
size_t dsa_sparse_attn_fwd_workspace_size(int B, int S, int H, int Hkv, int Dqk, int Dv);
int dsa_sparse_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* idx, int B,
                        int S, int H, int Hkv, int Dqk, int Dv, int k, float scale, void* O,
                        float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * dsa_sparse_attn_fwd_kernel - which kernel dsa_sparse_attn_fwd runs for a shape:
 * DSA_FWD_GATHER_TC (the gathered-key tensor-core kernel, one launch),
 * DSA_FWD_DENSE_TC (the dense-tile tensor-core kernel: a bitmap build and the
 * attention, two launches) or DSA_FWD_MMA_SYNC (one launch); the negated status
 * (-DSA_ERR_INVALID_ARG, -DSA_ERR_UNSUPPORTED) when the call would refuse the shape.
 * Launches nothing.
 */
#define DSA_FWD_GATHER_TC 0
#define DSA_FWD_DENSE_TC 1
#define DSA_FWD_MMA_SYNC 2
int dsa_sparse_attn_fwd_kernel(int B, int S, int H, int Hkv, int Dqk, int Dv, int k,
                               float scale);

/*
 * dsa_sparse_attn_fwd_dense - the same result from the dense-tile kernel only
 * (the pages' own design evaluates the masked logits as dense blocks with
 * partial mask blocks: "Support Ring Attention with DeepSeek DSA Sparse
 * Indexer", Forward Flow). Arguments, workspace included, as for
 * dsa_sparse_attn_fwd. Supported: any Hkv dividing H, 1 <= H <= 128, (Dqk, Dv)
 * in {(128, 128), (192, 128)}, S <= 65536, a positive scale; DSA_ERR_UNSUPPORTED
 * otherwise.
 */
int dsa_sparse_attn_fwd_dense(const void* Q, const void* K, const void* V, const int32_t* idx,
                              int B, int S, int H, int Hkv, int Dqk, int Dv, int k, float scale,
                              void* O, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * dsa_sparse_attn_bwd - gradients of the sparse attention ("Support Ring
 * Attention with DeepSeek DSA Sparse Indexer", Backward Flow step 6:
 * dQ = dP.K, dK = dP^T.Q, dV = P^T.dO over the same mask, "dP" being the
 * gradient of the logits):
 *
 *     P_j recomputed from lse;  Delta = sum_c dO[c] O[c];  dS_j = P_j (dO.V[s_j] - Delta)
 *     dQ[t,h] = scale sum_j dS_j K[s_j];  dK[s] = scale sum dS Q;  dV[s] = sum P dO
 *
 *   Q, K, V, idx as for the forward; O, lse the forward's outputs;
 *   dO bf16 [B, S, H, Dv];  dQ bf16 [B, S, H, Dqk] out;
 *   dK bf16 [B, S, Hkv, Dqk] out;  dV bf16 [B, S, Hkv, Dv] out;
 *   ws  workspace of dsa_sparse_attn_bwd_workspace_size() bytes, 16-byte aligned
 *       (overwritten): the fp32 dK/dV accumulators [B*S*Hkv, Dqk + Dv] rounded up
 *       to 256 bytes, then, whenever the dense-tile kernels can take the shape,
 *       their selection bitmap, tile flags and Delta (fp32 [B, S, H]).
 *
 * Supported shapes as for the forward. dK/dV are summed with fp32 atomics, so
 * their rounding order is not fixed from run to run.
 */
size_t dsa_sparse_attn_bwd_workspace_size(int B, int S, int H, int Hkv, int Dqk, int Dv);
int dsa_sparse_attn_bwd(const void* Q, const void* K, const void* V, const int32_t* idx,
                        const void* O, const float* lse, const void* dO, int B, int S, int H,
                        int Hkv, int Dqk, int Dv, int k, float scale, void* dQ, void* dK, void* dV,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * dsa_sparse_attn_bwd_dense - the same gradients from the dense-tile kernels only:
 * a dQ pass over (batch, head, query tile) items and a key-major dK / dV pass over
 * (batch, key tile, group of heads) items, both under the bitmap of the selection
 * (the pages' design: dense blocks with partial mask blocks and a key-major pass
 * for dK / dV, "Support Ring Attention with DeepSeek DSA Sparse Indexer",
 * Backward Flow). Arguments, workspace included, as for dsa_sparse_attn_bwd.
 * Supported: any Hkv dividing H, 1 <= H <= 128, (Dqk, Dv) in {(128, 128),
 * (192, 128)}, S <= 65536, a positive scale; DSA_ERR_UNSUPPORTED otherwise.
 * dsa_sparse_attn_bwd takes these kernels when they have fewer tile products for
 * the shape, and always for Hkv > 1; dsa_sparse_attn_bwd_noalloc never does (so
 * it takes Hkv = 1 only).
 */
int dsa_sparse_attn_bwd_dense(const void* Q, const void* K, const void* V, const int32_t* idx,
                              const void* O, const float* lse, const void* dO, int B, int S, int H,
                              int Hkv, int Dqk, int Dv, int k, float scale, void* dQ, void* dK, void* dV,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * dsa_sparse_attn_bwd_kernel - which kernels dsa_sparse_attn_bwd runs for a shape:
 * DSA_BWD_GATHER_TC (gathered-key tensor-core kernel + finalize: 2 launches),
 * DSA_BWD_DENSE_TC (bitmap, dQ pass, dK / dV pass, finalize: 4 launches) or
 * DSA_BWD_MMA_SYNC (2 launches); the negated status when the call would refuse the
 * shape. Launches nothing.
 */
#define DSA_BWD_GATHER_TC 0
#define DSA_BWD_DENSE_TC 1
#define DSA_BWD_MMA_SYNC 2
int dsa_sparse_attn_bwd_kernel(int B, int S, int H, int Hkv, int Dqk, int Dv, int k,
                               float scale);

/*
 * dsa_sparse_attn_bwd_noalloc - dsa_sparse_attn_bwd for callers that cannot
 * allocate device memory. The pages have no counterpart: this is a
 * deployment variant of the same backward pass, not part of the method.
 *
 * Callers that are handed their input and output buffers by a host program
 * and cannot obtain more device memory (a plugin inside a runtime that owns
 * every allocation through its own pool, or code that must not call
 * cudaMalloc while it runs because an allocation there can fail or stall the
 * device) cannot pass the fp32 workspace of dsa_sparse_attn_bwd. This entry
 * point takes the same tensors without it and keeps the dK/dV accumulator in
 * a fixed array inside the library: DSA_NOALLOC_BWD_MAX_FLOATS floats
 * (32 MiB), held on every GPU that loads the library until the process exits.
 *
 *  - Limit: B * S * Hkv * (Dqk + Dv) must not exceed DSA_NOALLOC_BWD_MAX_FLOATS
 *    (e.g. 26214 tokens at Dqk + Dv = 320); larger calls return
 *    DSA_ERR_WORKSPACE and launch nothing.
 *  - Nothing is allocated or freed. The first call on a device looks up the
 *    array's device address (cudaGetSymbolAddress) with that device current;
 *    make that first call before any stream capture.
 *  - Every call shares the one array and zeroes the part it uses before
 *    accumulating, so calls whose work overlaps on the GPU (two streams, or
 *    two host threads) race and corrupt each other's dK/dV. Serialise them.
 *  - Arguments, supported shapes and results are those of dsa_sparse_attn_bwd
 *    with Hkv = 1 (per-head K/V needs the dense-tile kernels, whose scratch is
 *    part of dsa_sparse_attn_bwd's workspace).
 */
#define DSA_NOALLOC_BWD_MAX_FLOATS 8388608
int dsa_sparse_attn_bwd_noalloc(const void* Q, const void* K, const void* V, const int32_t* idx,
                                const void* O, const float* lse, const void* dO, int B, int S,
                                int H, int Hkv, int Dqk, int Dv, int k, float scale, void* dQ,
                                void* dK, void* dV, void* stream);

/*
 * dsa_index_topk - dsa_index_scores followed by dsa_topk, fused through blocks of
 * query rows: the [B, S, S] score matrix never exists. Each block of block_rows
 * query rows is scored into a [B, block_rows, ld] fp32 buffer in `ws` (ld = S
 * rounded up to a multiple of 4) and its top-k is taken before the next block
 * reuses the buffer, so the scores' memory is B * block_rows * ld * 4 bytes instead
 * of B * S * ld * 4 (at S = 131072 and block_rows = 2048: 1 GiB instead of 64 GiB),
 * and a small block keeps them in L2. "DeepSeek3.2: Onboard sparse attention"
 * (Background: the top-k of the index scores gives the index mask) and "Implement QK
 * attention head chunking for CSA" (the dense score products run out of memory at
 * long context).
 *
 *   q_idx, k_idx, w, w_dtype, seg, B, S, Hi, Di as for dsa_index_scores;
 *   k, idx [B, S, k], count [B, S] (or NULL), vals [B, S, k] (or NULL) as for dsa_topk
 *               (identical results);
 *   block_rows  query rows per block: a positive multiple of 256;
 *   ws          at least dsa_index_topk_workspace_size(B, S, block_rows) bytes.
 *
 * Supported as for dsa_index_scores (bf16 inputs). DSA_ERR_WORKSPACE if ws is too small.
 */
size_t dsa_index_topk_workspace_size(int B, int S, int block_rows);
int dsa_index_topk(const void* q_idx, const void* k_idx, const void* w, int w_dtype,
                   const int32_t* seg, int B, int S, int Hi, int Di, int k, int block_rows,
                   int32_t* idx, int32_t* count, float* vals, void* ws, size_t ws_bytes,
                   void* stream);

/*
 * dsa_index_topk_fp8 - dsa_index_topk on e4m3 q_idx / k_idx with an optional
 * per-key scale of k: dsa_index_scores_fp8 followed by dsa_topk, through blocks of
 * query rows. Arguments as for dsa_index_topk, plus k_scale as for
 * dsa_index_scores_fp8 (Di a multiple of 16).
 */
int dsa_index_topk_fp8(const void* q_idx, const void* k_idx, const float* k_scale, const void* w,
                       int w_dtype, const int32_t* seg, int B, int S, int Hi, int Di, int k,
                       int block_rows, int32_t* idx, int32_t* count, float* vals, void* ws,
                       size_t ws_bytes, void* stream);

/*
 * dsa_index_topk_stream - dsa_index_scores followed by dsa_topk, with no score row in
 * memory (the streaming form of the fused indexer + top-k; "Implement QK attention head
 * chunking for CSA", Description: the dense score products do not fit at long context).
 * Results are those of dsa_index_topk, bit for bit.
 *
 *  1. A sampled indexer pass scores evenly spaced 128-key tiles of each query group's
 *     causal range: a 16th of its tiles, at least 8 and at most 32 (all of them when
 *     there are fewer).
 *  2. From each row's sample, a window [L, U) around its k-th largest score: the sample's
 *     order statistics at rank k * (sampled) / (valid keys), +- 5 standard deviations.
 *  3. The full indexer pass keeps, per row, the keys scoring >= U (their indices, in the
 *     row's idx slots, and with vals their scores in the row's vals slots) and the keys in
 *     [L, U) (index and score, up to 4096), and stores no other score. Rows with at most
 *     k keys take every valid key this way (U = L = -inf).
 *  4. Each row is settled from these two lists: when at most k keys score >= U and the
 *     two lists together hold at least min(k, valid keys), the k-th largest score lies in
 *     the window and is found there; ties go to the lower key index as in dsa_topk.
 *  5. A row the lists cannot settle (the sample misplaced its window, or a list
 *     overflowed) marks its block of block_rows query rows; such blocks are redone by
 *     dsa_index_topk's memory form (indexer and top-k of the block's scores in `ws`),
 *     launches that a flag on the device switches on. On typical score distributions few
 *     or no blocks are redone.
 *
 *   q_idx, k_idx, w, w_dtype, seg, B, S, Hi, Di, k, idx, count, vals: as for
 *               dsa_index_topk; vals needs k <= 2048 (the scores of a row are staged by
 *               slot in shared memory), DSA_ERR_UNSUPPORTED otherwise;
 *   block_rows  rows per redone block: a positive multiple of 256;
 *   ws          at least dsa_index_topk_stream_workspace_size(B, S, block_rows) bytes:
 *               the samples (16 KB per query row), the window lists (32 KB per query row)
 *               and one block of fp32 scores (B * block_rows * S * 4 bytes).
 *
 * Supported as for dsa_index_scores, with S <= 131072; DSA_ERR_UNSUPPORTED otherwise.
 */
size_t dsa_index_topk_stream_workspace_size(int B, int S, int block_rows);
int dsa_index_topk_stream(const void* q_idx, const void* k_idx, const void* w, int w_dtype,
                          const int32_t* seg, int B, int S, int Hi, int Di, int k, int block_rows,
                          int32_t* idx, int32_t* count, float* vals, void* ws, size_t ws_bytes,
                          void* stream);

/*
 * dsa_index_topk_stream_fp8 - dsa_index_topk_stream on e4m3 q_idx / k_idx with an optional
 * per-key scale of k (as dsa_index_scores_fp8; Di a multiple of 16).
 */
int dsa_index_topk_stream_fp8(const void* q_idx, const void* k_idx, const float* k_scale,
                              const void* w, int w_dtype, const int32_t* seg, int B, int S, int Hi,
                              int Di, int k, int block_rows, int32_t* idx, int32_t* count,
                              float* vals, void* ws, size_t ws_bytes, void* stream);

/*
 * dsa_indexer_loss - the indexer's auxiliary loss and its gradient with respect
 * to the index scores.
 *
 * "Implement QK attention head chunking for CSA" gives the target: every head's
 * attention scores go through an fp32 softmax over the valid tokens, are zeroed
 * elsewhere, summed over the heads and held constant. "Support Ring Attention
 * with DeepSeek DSA Sparse Indexer" (Loss Harvesting & Objective Injection) adds
 * the loss to the objective so that its gradient trains the indexer. The pages
 * do not print the loss itself; this library reads it as the KL divergence
 * between the head-averaged target and the softmax of the index scores, both
 * over the query's selected keys (slots j with 0 <= s_j = idx[b,t,j] <= t):
 *
 *   pbar_j = (1/H) sum_h exp(scale Q[b,t,h].K[b,s_j] - lse[b,t,h])
 *   q_j    = softmax_j(scores[b,t,s_j])
 *   kl[b,t]   = sum_j pbar_j (log pbar_j - log q_j)          (0 log 0 = 0)
 *   dI[b,t,j] = grad_scale (q_j - pbar_j)   (0 at slots without a selected key)
 *
 * dI is the gradient of grad_scale * sum_{b,t} kl[b,t] with respect to the score
 * at each slot: pass it to dsa_indexer_loss_bwd.
 *
 *   Q      bf16 [B, S, H, Dqk]     K    bf16 [B, S, Hkv, Dqk]
 *   idx    int32 [B, S, k]          lse  fp32 [B, S, H] (from dsa_sparse_attn_fwd)
 *   scores fp32 [B, S, ld_scores]   only the selected entries are read; or, with
 *          ld_scores = 0, fp32 [B, S, k]: the selected keys' scores slot by slot (the
 *          `vals` of dsa_topk / dsa_index_topk / dsa_index_topk_stream), read contiguously
 *   kl     fp32 [B, S] out          dI   fp32 [B, S, k] out
 *
 * Hkv divides H (head h reads K head h / (H / Hkv)). The tensor-core kernel takes
 * Hkv = 1, 1 <= H <= 128, Dqk in {128, 192} and scale > 0; every other shape runs on
 * the CUDA cores (one CTA per query row, far slower). Rows with no selected key get
 * kl = 0 and dI = 0. An index outside [-1, S) is skipped and
 * recorded as DSA_STAGE_LOSS | DSA_DEVERR_BAD_INDEX. kl is accumulated with
 * atomics (summation order unspecified).
 */
int dsa_indexer_loss(const void* Q, const void* K, const int32_t* idx, const float* lse,
                     const float* scores, int64_t ld_scores, int B, int S, int H, int Hkv,
                     int Dqk, int k, float scale, float grad_scale, float* kl, float* dI,
                     void* stream);

/*
 * dsa_indexer_loss_bwd - the gradient of the indexer loss with respect to the
 * indexer's inputs, given dI from dsa_indexer_loss. With
 * I[t,s] = sum_h w[t,h] max(0, z_h), z_h = q_idx[t,h].k_idx[s] (the index score
 * of dsa_index_scores) and the derivative of max(0, z) at z = 0 taken as 0:
 *
 *   dw[b,t,h]     = sum_j dI[b,t,j] max(0, z_hj)
 *   dq_idx[b,t,h] = sum_j dI[b,t,j] w[b,t,h] [z_hj > 0] k_idx[b,s_j]
 *   dk_idx[b,s]   = sum over (t, j) with s_j = s of sum_h dI[b,t,j] w[b,t,h] [z_hj > 0] q_idx[b,t,h]
 *
 * over the selected slots (0 <= s_j <= t).
 *
 *   q_idx  bf16 [B, S, Hi, Di]   k_idx bf16 [B, S, Di]   w fp32 [B, S, Hi]
 *   idx    int32 [B, S, k]       dI    fp32 [B, S, k]
 *   dq_idx fp32 [B, S, Hi, Di] out   dk_idx fp32 [B, S, Di] out   dw fp32 [B, S, Hi] out
 *
 * Hi = 64, Di = 128 run on the tensor cores, with G = dI w [z > 0] rounded to bf16
 * and fp32 accumulation; other shapes on the CUDA cores in fp32 (one CTA per query
 * row, far slower), up to Hi * (Di + 1) <= 51200 (DSA_ERR_UNSUPPORTED above). dk_idx
 * is accumulated with fp32 atomics (summation order unspecified).
 */
int dsa_indexer_loss_bwd(const void* q_idx, const void* k_idx, const float* w,
                         const int32_t* idx, const float* dI, int B, int S, int Hi, int Di,
                         int k, float* dq_idx, float* dk_idx, float* dw, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
