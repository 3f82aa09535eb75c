/*
 * gw.h - C ABI of the paged hybrid decode-attention library (GB300, sm_103a).
 *
 * The library computes one decode step of attention for a Gemma-4-style
 * hybrid stack, over paged KV pools, on the GPU:
 *
 *   - gw_kv_append           RoPE on the rotated slice of K, then page write
 *                            (optionally rounding to e4m3) of the step's rows.
 *   - gw_decode_attn_local   sliding-window attention, head dim 256, GQA.
 *   - gw_decode_attn_global  global attention, head dim 512, one KV head, over
 *                            the compressed V + k_rot pool (K rebuilt on chip)
 *                            or over a full K + V control pool.
 *
 * Sources of the operations (page title, section):
 *   [pegainfer] "Gemma 4" (pegainfer model page): intro, "Scheduling",
 *               "Architecture notes".  Five of six layers are sliding-window
 *               local attention at head dim 256 (window 1024, RoPE on all 256
 *               dims, theta 10k); every sixth layer and the last are global
 *               attention at head dim 512 with one KV head and a proportional
 *               RoPE on 128 of 512 dims (theta 1M, denominator 512).  Each
 *               kind has its own paged pool of 16-token pages; every active
 *               request advances one token per batched step and a new
 *               prompt's rows are computed in the same step.
 *   [Gewell]    "Gewell - Gemma4 inference engine", "the Why": K and V are
 *               tied on global layers and RoPE rotates 25% of K, so a token
 *               can be cached as V plus the rotated K slice (0.625x of K+V);
 *               K is rebuilt from V for the attention math.
 *   [PR1012]    "feat(gemma4): the sliding family serves an opt in fp8 KV
 *               pool", "Description": the sliding family's K/V may be stored
 *               as e4m3 at scale 1.0; the element type is an enum on the
 *               pool layout; entry points without an fp8 variant refuse a
 *               one-byte layout.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates, frees or synchronises; every call only
 *     enqueues work on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and returns.
 *   - Arguments are validated on the host before anything is launched.  A
 *     failure returns a non-zero gw_status and leaves a message, naming the
 *     entry point, in gw_last_error() (thread-local).
 *   - Values that live in device memory (slots, positions, lengths, page ids)
 *     are checked by the kernels: an out-of-range value skips the access it
 *     would have made and ORs a GW_DEV_* bit into *dev_status (a device int32
 *     the caller zeroes and reads when it wants; may be NULL).  Output rows of
 *     a sequence with out-of-range metadata are written as zeros.
 *   - bf16 is IEEE binary32 truncated to 16 bits; e4m3 is the OCP "e4m3fn"
 *     8-bit format (bias 7, max 448, no infinities).
 */
#ifndef GW_H
#define GW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
typedef int32_t gw_status;
#define GW_OK 0
#define GW_ERR_INVALID_ARG 1 /* null/misaligned pointer, bad size or geometry */
#define GW_ERR_UNSUPPORTED 2 /* valid but not implemented, e.g. e4m3 global  */
#define GW_ERR_WORKSPACE 3   /* workspace_bytes below gw_attn_workspace_bytes */
#define GW_ERR_CUDA 4        /* a launch failed; message has the CUDA error  */

/* bits a kernel ORs into *dev_status */
#define GW_DEV_SLOT_RANGE 1  /* append slot outside [0, num_pages*16)        */
#define GW_DEV_POS_RANGE 2   /* append position outside [0, max_pos)          */
#define GW_DEV_PAGE_RANGE 4  /* block-table entry outside [0, num_pages)      */
#define GW_DEV_LEN_RANGE 8   /* seq_len < rows, or > max_pages_per_seq * 16   */
#define GW_DEV_TIMEOUT 16    /* a bounded wait gave up (work abandoned)       */
#define GW_DEV_WORKSPACE 32  /* the step needs more split-KV partials than the
                                workspace was sized for (nothing computed)    */

/* ---- pool description --------------------------------------------------- */
#define GW_KV_BF16 0
#define GW_KV_E4M3 1

#define GW_LAYOUT_LOCAL 0         /* sliding-window layers                   */
#define GW_LAYOUT_GLOBAL_FOLDED 1 /* global layers, V(512) + k_rot(128)     */
#define GW_LAYOUT_GLOBAL_FULL 2   /* global layers, K(512) + V(512) control */
#define GW_LAYOUT_GLOBAL_FOLDED_E4M3 3 /* opt-in: V(512) + k_rot(128) in e4m3 */

/*
 * A paged KV pool: `num_pages` pages of 16 tokens at `base` (device, 256-byte
 * aligned).  A token lives at slot = page * 16 + offset.  Element order
 * inside a page:
 *
 *   LOCAL   (dtype bf16 or e4m3, head_dim 256, rot_dim 256, kv_heads >= 1)
 *           [kv_head][K=0 / V=1][token 16][dim 256]
 *           -> kv_heads * 16 KiB per page (bf16), kv_heads * 8 KiB (e4m3).
 *   GLOBAL_FOLDED (bf16, head_dim 512, rot_dim 128, kv_heads 1)
 *           a token row is the 640-vector  V[0:512] || k_rot[0:128],
 *           stored as [token block 2][column block 80][row 8][column 8]:
 *           token o = 8*tb + r, row element e = 8*cb + c.  20480 B per page.
 *   GLOBAL_FULL   (bf16, head_dim 512, rot_dim 128, kv_heads 1)
 *           a token row is K[0:512] || V[0:512], same 8x8 blocking with 128
 *           column blocks.  32768 B per page.
 *   GLOBAL_FOLDED_E4M3 (e4m3, head_dim 512, rot_dim 128, kv_heads 1)
 *           the folded row V[0:512] || k_rot[0:128] with every element
 *           rounded once to e4m3, stored as [token block 2][column block
 *           40][row 8][column 16]: token o = 8*tb + r, e = 16*cb + c.
 *           10240 B per page (0.3125x of GLOBAL_FULL).  The pages serve e4m3
 *           for the sliding family only and refuse it for global layers, so
 *           this layout is an explicit opt-in: dtype e4m3 on GLOBAL_FOLDED
 *           stays refused ("supports only local").
 *
 * In the folded layout the unrotated dims of K are not stored: attention uses
 * K = k_rot || V[128:512].  The caller folds the k_norm gain of those dims
 * into q (exact up to rounding order).
 */
typedef struct gw_kv_pool {
  int32_t layout;    /* GW_LAYOUT_* */
  int32_t dtype;     /* GW_KV_*     */
  void* base;        /* device pointer, 256-byte aligned */
  int64_t num_pages; /* >= 1 */
  int32_t page_size; /* must be 16 */
  int32_t kv_heads;  /* local: 1..64; global: 1 */
  int32_t head_dim;  /* local: 256; global: 512 */
  int32_t rot_dim;   /* local: 256; global: 128 */
} gw_kv_pool;

/* Bytes of one page of `pool`, 0 if the description is invalid (base may be
 * NULL here: the size is needed before the pool is allocated). */
size_t gw_pool_page_bytes(const gw_kv_pool* pool);

/*
 * gw_kv_append - write the step's K/V rows into `pool`.
 *
 * [pegainfer] "Architecture notes" (RoPE of each family; global K and V from
 * one projection), [Gewell] "the Why" (store V + rotated K slice),
 * [PR1012] "Description" (e4m3 at scale 1.0 for the sliding family).
 *
 *   k, v     bf16.  LOCAL: [num_rows][kv_heads][256].  GLOBAL: [num_rows][512]
 *            (FOLDED reads only k[:, 0:128]; FULL stores k[:, 128:512] as is).
 *   slot     int32 [num_rows]: page * 16 + offset of each row.
 *   pos      int32 [num_rows]: the row's absolute position (RoPE angle).
 *   rope_cs  float32 [max_pos][rot_dim/2][2]: (cos, sin) of pos * inv_f_i,
 *            inv_f_i = theta^(-2i / head_dim), computed in float64 and
 *            rounded once to float32.
 *
 * For i in [0, rot_dim/2), with x0 = k[i], x1 = k[i + rot_dim/2] (exact
 * fp32 of the bf16 inputs) and (c, s) = rope_cs[pos][i], the stored rotated
 * pair is  r0 = fl(fl(x0*c) - fl(x1*s)),  r1 = fl(fl(x1*c) + fl(x0*s))
 * (binary32, no fused multiply-add), then rounded once to the pool type:
 * bf16 round-to-nearest-even, or e4m3 round-to-nearest-even saturating to
 * +-448.  V (and the unrotated K dims of a FULL pool) are copied (bf16) or
 * rounded once to e4m3 (a GLOBAL_FOLDED_E4M3 pool rounds k_rot once from its
 * float32 rotation and V once from bf16).  Rows whose slot or pos is out of
 * range are skipped
 * (GW_DEV_SLOT_RANGE / GW_DEV_POS_RANGE).  num_rows == 0 is a no-op.
 * rope_cs is the table gw_rope_cs fills.
 * Alignment: k, v, rope_cs 16 B; slot, pos 4 B.
 * Errors: GW_ERR_INVALID_ARG, GW_ERR_UNSUPPORTED (e4m3 on a GLOBAL_FOLDED or
 * GLOBAL_FULL pool: "supports only local"), GW_ERR_CUDA.
 */
gw_status gw_kv_append(const gw_kv_pool* pool, const void* k, const void* v, int32_t num_rows,
                       const int32_t* slot, const int32_t* pos, const float* rope_cs, int32_t max_pos,
                       int32_t* dev_status, void* stream);

/*
 * gw_rope_cs - fill the (cos, sin) table that gw_kv_append takes as rope_cs.
 *
 * [pegainfer] "Architecture notes": local layers rotate all 256 dims of K
 * with theta 10k; global layers use a proportional RoPE that rotates 128 of
 * the 512 dims with theta 1M while the frequency denominator stays the full
 * head dim.  So the table takes both the rotated width and the head dim:
 *
 *   inv_f_i = theta^((-2 i) / head_dim),      i in [0, rot_dim / 2)
 *   rope_cs[p][i] = (cos(p * inv_f_i), sin(p * inv_f_i)),  p in [0, max_pos)
 *
 * computed on the GPU in float64 (frequency, angle, cosine and sine) and
 * rounded once to float32.  Local pools take (theta 1e4, rot_dim 256,
 * head_dim 256); global pools (theta 1e6, rot_dim 128, head_dim 512).
 *
 *   rope_cs   device float32 [max_pos][rot_dim / 2][2], caller-owned,
 *             16-byte aligned; fully overwritten.
 * Errors: GW_ERR_INVALID_ARG (NULL or misaligned rope_cs, theta not finite
 * and positive, rot_dim odd or outside [2, head_dim], max_pos < 1),
 * GW_ERR_CUDA.  Asynchronous on `stream`.
 */
gw_status gw_rope_cs(float* rope_cs, double theta, int32_t rot_dim, int32_t head_dim, int32_t max_pos,
                     void* stream);

/*
 * gw_decode_attn_local - sliding-window attention on a LOCAL pool.
 *
 * [pegainfer] "Architecture notes", "Scheduling".  Sequence b holds tokens
 * [0, seq_lens[b]) (after this step's append) and contributes
 * n_b = cu_q_rows[b+1] - cu_q_rows[b] query rows, at positions
 * p = seq_lens[b] - n_b + r.  Row r of q head h attends to keys
 * j in [max(0, p - window + 1), p] of KV head h / (num_q_heads / kv_heads):
 *
 *   o = sum_j softmax_j(scale * q . K_j) V_j      (fp32 accumulation)
 *
 * Rows with n_b == 1 take the split-KV decode kernel (partials in
 * `workspace`, then a log-sum-exp combine); rows of sequences with n_b > 1
 * (prompt rows of a mixed step) take the causal prompt-row kernel.  The split
 * plan of a sequence depends only on its own length, so its result is
 * bit-identical whatever else is in the batch.
 *
 *   q, out       bf16 [total_rows][num_q_heads][256], total_rows = cu_q_rows[batch].
 *   cu_q_rows    int32 [batch+1], non-decreasing, cu_q_rows[0] = 0.
 *   seq_lens     int32 [batch].
 *   block_table  int32 [batch][max_pages_per_seq]: physical page of each
 *                logical page; entries before the window may be anything.
 *   max_q_rows   host bound on n_b (1 for a pure decode step).
 *   window       >= 1 (1024 for the served model).
 *   workspace    device scratch of at least gw_attn_workspace_bytes(...),
 *                256-byte aligned; contents need no initialisation.
 * On an e4m3 pool ([PR1012] "Description", "Verification": the sliding
 * family's fp8 pool serves decode and mixed steps alike) the contractions of
 * decode and prompt rows run on the e4m3 tiles as stored; each q row and
 * softmax weight enters as a sum of two e4m3 terms (q after an exact
 * power-of-two scaling per head or row), which carries it at about bf16
 * precision for any q whose logits are finite in fp32.
 *
 * Errors: GW_ERR_INVALID_ARG, GW_ERR_WORKSPACE, GW_ERR_UNSUPPORTED
 * (num_q_heads / kv_heads not in {1,2,4,8}; batch > 4096, since the decode
 * kernel keeps the batch's split plan in shared memory), GW_ERR_CUDA.
 * Every error but GW_ERR_CUDA is returned before anything is launched.
 */
gw_status gw_decode_attn_local(const gw_kv_pool* pool, const void* q, void* out, int32_t num_q_heads,
                               int32_t batch, const int32_t* cu_q_rows, const int32_t* seq_lens,
                               const int32_t* block_table, int32_t max_pages_per_seq, int32_t max_q_rows,
                               int32_t window, float scale, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream);

/*
 * gw_append_decode_attn_local - a decode step's append and attention in one
 * call: the same result as gw_kv_append of each decode row's K/V followed by
 * gw_decode_attn_local with max_q_rows = 1.
 *
 * [pegainfer] "Scheduling" (every active request advances one token per
 * batched step) and "Architecture notes" (local RoPE over all 256 dims,
 * theta 10k).  Sequence b with one row (cu_q_rows[b+1] - cu_q_rows[b] == 1)
 * appends k[r], v[r] (r = cu_q_rows[b]; [rows][kv_heads][256] bf16) at
 * position pos = seq_lens[b] - 1, in page block_table[b][pos / 16] at offset
 * pos % 16 - the slot and pos gw_kv_append would be given - with
 * gw_kv_append's rotation and rounding, so the pool holds the same bytes;
 * then that row attends over its window, the new key included.  Sequences
 * without a row are skipped.  The kernel that decodes a KV head's last chunk
 * writes its row before reading that page, so no second kernel and no
 * wait between the two.  rope_cs and max_pos as for gw_kv_append.  A row
 * with pos >= max_pos is not written (GW_DEV_POS_RANGE); a bad page entry is
 * reported as by gw_decode_attn_local.  bf16 and e4m3 pools.
 * Errors: those of gw_decode_attn_local; GW_ERR_INVALID_ARG (k, v, rope_cs
 * NULL or not 16-byte aligned, max_pos < 1).
 */
gw_status gw_append_decode_attn_local(const gw_kv_pool* pool, const void* k, const void* v, const float* rope_cs,
                                      int32_t max_pos, const void* q, void* out, int32_t num_q_heads, int32_t batch,
                                      const int32_t* cu_q_rows, const int32_t* seq_lens, const int32_t* block_table,
                                      int32_t max_pages_per_seq, int32_t window, float scale, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * gw_decode_attn_global - global attention on a GLOBAL_FOLDED, GLOBAL_FULL or
 * GLOBAL_FOLDED_E4M3 pool: as gw_decode_attn_local with no window
 * (j in [0, p]) and head dim 512.
 *
 * [pegainfer] "Architecture notes"; [Gewell] "the Why".  On a folded pool the
 * kernel forms K_j = k_rot_j || V_j[128:512] on chip from the same page tile
 * that supplies V_j.  num_q_heads must be 8, 16 or 32 and batch at most
 * 4096.  Errors as above; GW_ERR_UNSUPPORTED for dtype e4m3 on a GLOBAL_FOLDED
 * or GLOBAL_FULL pool ("supports only local"), and for prompt rows
 * (max_q_rows > 1) on a GLOBAL_FOLDED_E4M3 pool.
 *
 * On a GLOBAL_FOLDED_E4M3 pool the contractions run on the e4m3 tiles as
 * stored; q and the softmax weights enter them as sums of two e4m3 terms
 * (q after an exact per-head power-of-two scaling), which carries them at
 * about bf16 precision.  Output rows match attention over the stored e4m3
 * values within the same tolerance as a bf16 pool.
 */
gw_status gw_decode_attn_global(const gw_kv_pool* pool, const void* q, void* out, int32_t num_q_heads,
                                int32_t batch, const int32_t* cu_q_rows, const int32_t* seq_lens,
                                const int32_t* block_table, int32_t max_pages_per_seq, int32_t max_q_rows,
                                float scale, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                void* stream);

/*
 * gw_append_decode_attn_global - a decode step's append and attention on a
 * global pool in one call: the same result as gw_kv_append of each decode
 * row's k, v (GLOBAL shapes, [rows][512] bf16) followed by
 * gw_decode_attn_global with max_q_rows = 1.
 *
 * [pegainfer] "Scheduling" and "Architecture notes" (global RoPE on 128 of
 * 512 dims, theta 1M, denominator 512); [Gewell] "the Why" (the folded row).
 * Each sequence with one row appends it at pos = seq_lens[b] - 1 as
 * gw_append_decode_attn_local does; the kernel that decodes the sequence's
 * last chunk writes the row before copying the tile that holds it.  All
 * three global layouts.  Errors: those of gw_decode_attn_global;
 * GW_ERR_INVALID_ARG (k, v, rope_cs NULL or not 16-byte aligned,
 * max_pos < 1).
 */
gw_status gw_append_decode_attn_global(const gw_kv_pool* pool, const void* k, const void* v, const float* rope_cs,
                                       int32_t max_pos, const void* q, void* out, int32_t num_q_heads, int32_t batch,
                                       const int32_t* cu_q_rows, const int32_t* seq_lens, const int32_t* block_table,
                                       int32_t max_pages_per_seq, float scale, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * gw_decode_attn_global_lse - gw_decode_attn_global for decode rows
 * (max_q_rows 1) that also writes each row's log-sum-exp:
 *
 *   lse[row][h] = ln( sum_j exp(scale * q_h . K_j) )      over the row's keys
 *
 * (-inf for a row without keys), float32 [total_rows][num_q_heads],
 * 4-byte aligned, caller-owned.  With it, attention over a long sequence
 * whose keys are spread over several pools (one per rank of a
 * context-parallel split, each pool holding a contiguous range of the
 * sequence's pages, renumbered from 0) is the gw_merge_lse of the per-range
 * results: the split-KV combine applied across ranks.  The pages run one GPU
 * per sequence; this is the multi-GPU extension of the same split.
 * Errors as gw_decode_attn_global; GW_ERR_INVALID_ARG for a NULL lse.
 */
gw_status gw_decode_attn_global_lse(const gw_kv_pool* pool, const void* q, void* out, float* lse,
                                    int32_t num_q_heads, int32_t batch, const int32_t* cu_q_rows,
                                    const int32_t* seq_lens, const int32_t* block_table, int32_t max_pages_per_seq,
                                    float scale, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    void* stream);

/*
 * gw_merge_lse - merge n_parts attention results of the same rows computed
 * over disjoint key sets (the ranks of a context-parallel split), by their
 * log-sum-exp:
 *
 *   M = max_r lse_r,  w_r = exp(lse_r - M),
 *   out = (sum_r w_r o_r) / (sum_r w_r),   lse_out = M + ln(sum_r w_r),
 *
 * in float32 with the parts added in order r = 0, 1, ... (a part whose lse
 * is -inf contributes nothing and its o is not read; a row whose parts are
 * all -inf is written as zeros).
 *   o_parts     host array of n_parts device pointers, each bf16
 *               [rows][num_heads][head_dim], 16-byte aligned.
 *   lse_parts   host array of n_parts device pointers, each float32
 *               [rows][num_heads], 4-byte aligned.
 *   out         bf16 [rows][num_heads][head_dim], 16-byte aligned.
 *   lse_out     float32 [rows][num_heads] or NULL.
 *   n_parts in [1, 16]; head_dim 256 or 512.
 * Errors: GW_ERR_INVALID_ARG, GW_ERR_CUDA.  Asynchronous on `stream`.
 */
gw_status gw_merge_lse(int32_t n_parts, const void* const* o_parts, const float* const* lse_parts, void* out,
                       float* lse_out, int32_t rows, int32_t num_heads, int32_t head_dim, void* stream);

/*
 * Workspace bytes an attention call on `pool` needs for `batch` sequences of
 * at most `max_seq_len` tokens and `max_q_rows` rows each (window ignored for
 * global pools).  0 on an invalid description.
 */
size_t gw_attn_workspace_bytes(const gw_kv_pool* pool, int32_t num_q_heads, int32_t batch,
                               int32_t max_seq_len, int32_t max_q_rows, int32_t window);

/*
 * gw_decode_attn_local_noalloc - gw_decode_attn_local without a workspace
 * argument, for callers that cannot allocate device memory when they run
 * attention (an embedding runtime without a device allocator of its own, a
 * host that forbids device allocation once serving has started).  The pages
 * this library follows have no counterpart of this entry point; it exists
 * only for such callers.
 *
 * Same arguments, semantics, results and errors as gw_decode_attn_local,
 * minus workspace/workspace_bytes.  The split-KV scratch is a file-scope
 * device array of gw_noalloc_scratch_bytes() = 32 MiB that every GPU loading
 * this library keeps until the process exits; the call allocates and frees
 * nothing.  Arguments are checked as by gw_decode_attn_local (same statuses
 * for the same faults); a call whose gw_attn_workspace_bytes(...) (with
 * max_seq_len = max_pages_per_seq * 16) exceeds 32 MiB returns
 * GW_ERR_WORKSPACE, before anything is launched.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress) and caches it with the current CUDA
 * context; a call in another context (after a device reset) looks it up
 * again.  Make the first call on each device before any stream capture.  All calls share the one array and it keeps the
 * last call's contents (each call re-initialises what it needs), so calls
 * whose executions overlap on the GPU (different streams without ordering)
 * race on it.  Sequences with more than one query row (prompt rows of a mixed
 * step) are served as by gw_decode_attn_local, within the same 32 MiB.
 */
gw_status gw_decode_attn_local_noalloc(const gw_kv_pool* pool, const void* q, void* out, int32_t num_q_heads,
                                       int32_t batch, const int32_t* cu_q_rows, const int32_t* seq_lens,
                                       const int32_t* block_table, int32_t max_pages_per_seq, int32_t max_q_rows,
                                       int32_t window, float scale, int32_t* dev_status, void* stream);

/* Bytes of the static scratch behind gw_decode_attn_local_noalloc. */
size_t gw_noalloc_scratch_bytes(void);

/*
 * gw_set_max_ctas - cap the CTAs of the attention kernels that the calling
 * thread launches from now on (0 = one per SM, the default); appends then
 * launch at most 16 CTAs per allowed SM.
 *
 * [pegainfer] "Async prefill lane": a new prompt's prefill runs on its own
 * stream while decode goes on, capped at a share of the SMs so that it
 * cannot take the whole GPU.  The decode and prompt-row kernels here are
 * persistent with one CTA per SM (their shared memory allows no second), and
 * deal their work round-robin over the CTAs they have, so a CTA cap is an SM
 * cap: a prefill lane launched with a cap of N and a decode lane with the
 * SM count minus N run side by side on disjoint SMs.  Results do not depend
 * on the cap (a work unit's arithmetic never depends on which CTA runs it).
 * The setting is per host thread and is read when a call launches (for a
 * CUDA graph: when it is captured).
 * Errors: GW_ERR_INVALID_ARG (max_ctas < 0).
 */
gw_status gw_set_max_ctas(int32_t max_ctas);

/*
 * gw_set_early_launch - whether the calling thread's later launches may
 * start while the previous kernel of their stream is still running (1, the
 * default: programmatic dependent launch, whose early CTAs wait on chip for
 * their predecessor) or only once it has finished (0).  A capped prefill
 * lane beside a decode lane should use 0: its early CTAs, waiting out a long
 * prompt kernel, would otherwise hold registers and threads on the decode
 * lane's SMs and keep its kernels from starting.  Never an error.
 */
gw_status gw_set_early_launch(int32_t on);

/*
 * gw_set_early_inputs - whether the calling thread's later decode-attention
 * calls may read their index inputs before the previous kernel of their
 * stream has finished (1) or only after it (0, the default).
 *
 * With programmatic dependent launch a decode kernel starts while its
 * predecessor (typically this layer's gw_kv_append, or the previous layer's
 * combine) is still running, and waits on chip before touching anything that
 * predecessor may write.  With 1, the decode kernels compute their split plan
 * from cu_q_rows and seq_lens and fetch their first units' block-table
 * entries before that wait, which takes two dependent round trips off the
 * call; gw_kv_append likewise reads slot, pos and the RoPE table rows they
 * select before its wait, and a gw_append_decode_attn_local call the length,
 * page and RoPE rows of the first row it appends.  KV pages, q, k, v, the workspace, out and
 * dev_status are still touched only after the wait.  The caller promises
 * that the kernel just before each call in its stream does not write that
 * call's cu_q_rows, seq_lens, block_table, slot, pos or rope_cs, as holds
 * when they are uploaded for the whole step before its first layer.  Results
 * do not depend on the setting.  Read when a call launches (for a CUDA
 * graph: when it is captured).  Never an error.
 */
gw_status gw_set_early_inputs(int32_t on);

/*
 * gw_bw_probe - a measurement aid, not part of the method: streams the first
 * floor(bytes / 8192) * 8192 bytes of the device buffer `buf` through a
 * bulk-copy pipeline (one CTA per SM, 8 warps, each with a 2-stage ring of
 * 8 KiB shared-memory stages filled by two 4 KiB cp.async.bulk copies; the
 * global decode kernel copies its pages with the same instruction) and
 * discards them, so that its rate is the read bandwidth such a pipeline can
 * reach on the GPU.  The pages this library
 * follows have no counterpart of this entry point.
 *   buf          device memory, 16-byte aligned, caller-owned, only read.
 *   bytes        >= 8192.
 *   dev_status   optional; GW_DEV_TIMEOUT if a copy never lands.
 * Errors: GW_ERR_INVALID_ARG (NULL or misaligned buf, bytes < 8192),
 * GW_ERR_CUDA.  Asynchronous on `stream`.
 */
gw_status gw_bw_probe(const void* buf, size_t bytes, int32_t* dev_status, void* stream);

/*
 * gw_bw_probe_tma - as gw_bw_probe, through the copy pipeline of the bf16
 * local decode kernel instead (the e4m3 one copies 2 KiB boxes of one K or V
 * chunk, which its tensor-core operands need contiguous):
 * one CTA per SM, 6 warps, each with a 2-stage
 * ring of 16 KiB shared-memory stages, a stage being one 16-token page head
 * (K then V) brought by 4 tensor-map copies of 4 KiB (one 128-byte chunk of
 * its 16 K and 16 V rows each, 128-byte swizzled).
 * The first floor(bytes / 16384) * 16384 bytes of `buf` are read as the
 * pages of a LOCAL bf16 pool with one KV head, in page order, and discarded.
 * A measurement aid with no counterpart in the pages.
 *   buf          device memory, 256-byte aligned, caller-owned, only read.
 *   bytes        in [16384, 2^36].
 * Errors: GW_ERR_INVALID_ARG, GW_ERR_CUDA.  Asynchronous on `stream`.
 */
gw_status gw_bw_probe_tma(const void* buf, size_t bytes, int32_t* dev_status, void* stream);

/*
 * gw_wait_selftest - a test aid, not part of the method: runs the bounded
 * mbarrier wait that every kernel of this library uses, on one warp, with a
 * limit of `limit_ns` instead of the kernels' 2 s.  A phase that an arrival
 * completes is waited on first (must succeed); then a phase that nothing
 * ever completes, whose wait must give up after limit_ns, OR GW_DEV_TIMEOUT
 * into *dev_status and return, so that the kernel ends normally and the
 * context stays usable.  This is how the kernels' timeout path is tested
 * without hanging a GPU.  The pages this library follows have no
 * counterpart of this entry point.
 *   dev_status  device int32, caller-zeroed.
 *   result      device int32[3]: {first wait succeeded (1), second wait gave
 *               up (1), microseconds spent in the second wait}.
 *   limit_ns    in [1e3, 1e9].
 * Errors: GW_ERR_INVALID_ARG, GW_ERR_CUDA.  Asynchronous on `stream`.
 */
gw_status gw_wait_selftest(int32_t* dev_status, int32_t* result, int64_t limit_ns, void* stream);

/* Message of the calling thread's last failed call ("" if none). */
const char* gw_last_error(void);

/* ABI version of this library. */
int32_t gw_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GW_H */
