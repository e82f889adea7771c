/*
 * oscar.h -- C ABI of liboscar: the decode hot path of OScaR (Omni-Scaled
 * Canalized Rotation) INT2 KV-cache quantisation, for NVIDIA GB300 (sm_103a).
 *
 * Sources (page title and section):
 *  [rainbus] "OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀" (paper.rainbus.top
 *            summary): 方法步骤详情 (method step details), 前置知识, 论文图表 Fig. 2.
 *  [notes]   "OScaR: The Occam's Razor for Extreme KV Cache Quantization in LLMs
 *            and Beyond" (reading notes): II. Method -- Step One: Canalized
 *            Rotation; Step Two: Omni-Token Scaling; End-to-End Flow.
 *            III. Experiments -- Efficiency.
 *  [news]    news article on arXiv 2605.19660 (animattoys.com): 二 (the two
 *            steps), 三 (three kernels; packed cache and residual cache).
 *
 * Conventions (all calls)
 *  - head_dim D = 128, key block G = 32 tokens, residual window R = 128 tokens.
 *  - Every data pointer is DEVICE memory owned by the caller.  The library
 *    never allocates or frees memory and keeps no state except one device
 *    status word (read with oscar_device_status) and a host launch counter.
 *  - Pointers must be 16-byte aligned (else OSCAR_ERR_ALIGNMENT).
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *    stream).  Arguments are validated on the host before any launch; a
 *    validation failure launches nothing and leaves the cache struct unchanged.
 *    A launch failure returns OSCAR_ERR_CUDA.  Kernels that hit an internal
 *    wait limit record it in the device status word instead of hanging.
 *  - bf16 / fp16 values are passed as their 16-bit patterns.
 *  - (b, h) rows are contiguous: "[B][Hkv][X]" means row (b*Hkv + h) of X.
 *  - Query head j reads KV head j / g where g = Hq / Hkv (grouped-query
 *    attention); g is any whole number from 1 to 16 (Hq a multiple of Hkv).
 *    The decode kernels work 1, 2, 4 or 8 query heads per (b, h) CTA: a
 *    group of 3 runs as 4 heads with one padding head, groups of 5 to 7 as
 *    8, and groups of 9 to 16 as two slices of 8 per KV head, each reading
 *    the KV head's cache (padding heads are computed, never written).
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t oscar_bf16;
typedef uint16_t oscar_f16;

typedef enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad flag, state violation */
  OSCAR_ERR_UNSUPPORTED = 2,   /* e.g. Hq/Hkv not a whole number in 1..16 */
  OSCAR_ERR_ALIGNMENT = 3,     /* pointer not 16-byte aligned */
  OSCAR_ERR_CAPACITY = 4,      /* would write past T_cap */
  OSCAR_ERR_WORKSPACE = 5,     /* workspace too small or null */
  OSCAR_ERR_CUDA = 6,          /* a CUDA runtime call failed */
  OSCAR_ERR_DEVICE_STATUS = 7  /* a kernel recorded an error (see oscar_device_status) */
} oscar_status;

/* Ablation flags ([notes] III, Ablations: rotation only / scaling only).
 * 0 = the method: rotation then scaling, each token-head's key scaled by its
 * own norm.
 * OSCAR_NORM_ALL_HEADS: norm-scope variant.  The norm of token i is taken over
 * the rotated keys of all Hkv heads together ([notes] II, Notation: k_i in
 * R^{H*d_h} with n_i = ||k_i||; Step Two: "across all heads"), every head's
 * key is divided by it, and each head stores the same norm.  A head's k_hat
 * then has norm <= 1 rather than 1. */
enum { OSCAR_NO_ROTATE = 1u, OSCAR_NO_SCALE = 2u, OSCAR_NORM_ALL_HEADS = 4u };

/* Target norm (the scaling target whose choice [rainbus] 独立分析的弱点 (1)
 * says an appendix ablates): keys are scaled to norm `target` instead of 1 and
 * the stored norm is n / target, so dequantisation is unchanged.  0 means 1.
 * Accepted range [2^-8, 2^8].  A power of two changes no code (the min-max
 * quantiser is scale-equivariant and such a product is exact); other values
 * move the bf16 / fp16 roundings. */

#define OSCAR_HEAD_DIM 128
#define OSCAR_GROUP 32
#define OSCAR_RESIDUAL 128

/*
 * The KV cache of one attention layer for B sequences and Hkv KV heads:
 * the "packed cache" of INT2 codes, quantisation parameters and token-norm
 * tags plus the "residual cache" of the newest <= 128 tokens in 16 bit
 * ([news] 三; [rainbus] Fig. 2(c)).  Plain old data; every pointer is caller
 * device memory.  n_packed and n_res are uniform across the batch and are
 * advanced by the calls below (host-side bookkeeping).
 *
 * Packed layout: one record of OSCAR_BLOCK_BYTES per block of 32 tokens,
 * records [B][Hkv][T_cap/32] contiguous (T_cap a multiple of 32).  The
 * record takes the place of separate key-code, value-code, step, zero and
 * norm arrays: one 1-D bulk copy brings a whole block into shared memory.
 * Byte offsets inside a record:
 *     0  key codes    uint32 [32 tokens][8]: 16 codes per word; word w of a
 *                     token holds channels 16w..16w+15, channel 16w+j at bit
 *                     2*(j/2) + 16*(j%2) (even channels in the low half-word,
 *                     odd channels in the high half-word)
 *  1024  value codes  uint32 [256]: word 128*kh + 4*(4g+t) + 2p + hh (kh, p, hh
 *                     in {0,1}, g in 0..7, t in 0..3) holds token 16kh+2t+8p
 *                     in its low half-word and the next token in its high
 *                     half-word; slot k (bits 2k..2k+1 of a half) holds channel
 *                     g + 8*(8hh+k)
 *  2048  key step     fp16 [128] per channel ([rainbus] 方法步骤详情 (2), G = 32)
 *  2304  key zero     fp16 [128] per channel
 *  2560  key norms    fp16 [32] per token ([notes] Step Two)
 *  2624  value step   fp16 [32] per token
 *  2688  value zero   fp16 [32] per token
 *        (the three per-token arrays hold token t of the block at position
 *        4*(t%8) + t/8, so that tokens i, i+8, i+16, i+24 sit together)
 * Residual layout:
 *  k_res    bf16 [B][Hkv][128][128] rotated, unit-norm keys (slot = age order)
 *  v_res    bf16 [B][Hkv][128][128] values
 *  k_res_norm fp16 [B][Hkv][128]
 * Codes c in {0,1,2,3} dequantise to c*step + zero (x norm for keys).
 */
#define OSCAR_BLOCK_BYTES 2752

/*
 * INT4 option (cache field bits = 4; the pages fix only INT2, [rainbus]
 * 局限与改进 (1) names other widths as unstudied): the same quantiser with
 * (max - min)/15 as the step and codes 0..15, in a 4800-byte record:
 *     0  key codes    u32 [32][16]: channel 8w+j at bit 4*(j/2) + 16*(j%2)
 *  2048  value codes  u32 [512]: word 256*kh + 128p + 4*(4g+t) + hh holds, in
 *                     its low half, token 16kh + 2t + 8p and in its high half
 *                     the next token; slot k (bits 4k..4k+3) is channel
 *                     g + 8*(4hh + k)
 *  4096  key step, 4352 key zero, 4608 key norms, 4672 value step,
 *  4736 value zero (as in the INT2 record)
 */
#define OSCAR_BLOCK_BYTES_INT4 4800

typedef struct {
  int B, Hkv, T_cap;
  uint8_t* packed;       /* [B][Hkv][T_cap/32] records (OSCAR_BLOCK_BYTES, INT4: _INT4) */
  oscar_bf16* k_res;
  oscar_bf16* v_res;
  oscar_f16* k_res_norm;
  int n_packed;      /* quantised tokens per row, multiple of the key group */
  int n_res;         /* residual tokens per row, 0..128 */
  unsigned flags;    /* OSCAR_NO_ROTATE / OSCAR_NO_SCALE / OSCAR_NORM_ALL_HEADS, fixed for the cache's life */
  float norm_target; /* target norm of the scaled keys (0 = 1), fixed for the cache's life */
  int key_group;     /* tokens sharing a key channel's step and zero: 32 (0), 64 or 128;
                        n_packed and every quantised run are multiples of it */
  int bits;          /* code width: 2 (0, the method) or 4; records of
                        OSCAR_BLOCK_BYTES or OSCAR_BLOCK_BYTES_INT4 */
} oscar_cache;

/*
 * Paged variant for batches whose sequences have different lengths (a
 * serving engine's layout; the pages have no counterpart in the method,
 * which is unchanged).  The packed cache lives in pages of 32 tokens: page p
 * holds one record (layout above) per KV head, record h at
 * pages + (p*Hkv + h)*OSCAR_BLOCK_BYTES (INT4: _INT4).  Logical block j of sequence b
 * (its tokens 32j..32j+31) is page block_table[b*max_blocks + j]; the
 * caller owns the page pool and the table and must map a block before a
 * call writes it.  Lengths are per sequence and live in device memory, so a
 * step needs no host round trip:
 *  n_packed[b]  quantised tokens of sequence b (multiple of the key group)
 *  n_res[b]     its residual tokens, 0..128
 * The residual window stays per (b, h) as in oscar_cache.
 */
typedef struct {
  int B, Hkv;
  int max_blocks;           /* row length of block_table */
  int n_pages;              /* pages in the pool (page ids 0..n_pages-1) */
  uint8_t* pages;           /* [n_pages][Hkv] records of OSCAR_BLOCK_BYTES */
  int32_t* block_table;     /* device [B][max_blocks] page ids (B * max_blocks < 2^31) */
  int32_t* n_packed;        /* device [B] */
  int32_t* n_res;           /* device [B] */
  oscar_bf16* k_res;        /* [B][Hkv][128][128] */
  oscar_bf16* v_res;        /* [B][Hkv][128][128] */
  oscar_f16* k_res_norm;    /* [B][Hkv][128] */
  unsigned flags;
  float norm_target;
  int key_group;            /* as in oscar_cache */
  int bits;                 /* as in oscar_cache; a page holds Hkv records of its size */
} oscar_paged_cache;

/*
 * Canalized Rotation of the queries: q' = H q with H the 128x128 Sylvester
 * Hadamard matrix scaled by 1/sqrt(128), applied online every decode step so
 * that q'.k' = q.k ([notes] Step One, "Query-side symmetric processing";
 * [rainbus] 方法步骤详情 (1)).  The softmax scale is not applied here.
 *  q      bf16 [B][Hq][128]   input
 *  q_rot  fp32 [B][Hq][128]   output (may not alias q)
 *  flags  OSCAR_NO_ROTATE copies q (as fp32); OSCAR_NO_SCALE has no effect.
 */
oscar_status oscar_rotate_q(const oscar_bf16* q, float* q_rot, int B, int Hq,
                            unsigned flags, void* stream);

/*
 * Canalized Rotation + Omni-Token Scaling of keys (the fused kernel (1) of
 * [news] 三): k' = H k, s = sum(k'^2), k_hat = k' * rsqrt(s) (hardware rsqrt,
 * [news] 三), norm = ||k|| ([notes] Step Two: divide each token by its own L2
 * norm and keep the norm).  A zero key gives k_hat = 0, norm = 0.
 * OSCAR_NO_ROTATE skips H; OSCAR_NO_SCALE keeps k' and writes norm = 1.
 * OSCAR_NORM_ALL_HEADS: s sums over the token's keys in all Hkv heads (the
 * sum is formed from the raw keys, 128 * sum(k^2) = sum(k'^2) by
 * orthogonality).  norm_target t (0 = 1): k_hat = t * k' * rsqrt(s) and
 * norm = ||k|| / t.
 *  k        bf16 input,  element (b,h,t,c) at k[((b*Hkv+h)*in_T + t)*128 + c], t < n_tok
 *  k_hat    bf16 output, element at k_hat[((b*Hkv+h)*out_T + out_t0 + t)*128 + c]
 *  norm_out fp16 output, element at norm_out[(b*Hkv+h)*out_T + out_t0 + t]
 * Requires n_tok >= 1, in_T >= n_tok, out_t0 + n_tok <= out_T.
 */
oscar_status oscar_rotate_scale_k(const oscar_bf16* k, int in_T,
                                  oscar_bf16* k_hat, oscar_f16* norm_out, int out_T, int out_t0,
                                  int B, int Hkv, int n_tok, unsigned flags, float norm_target,
                                  void* stream);

/*
 * Quantisation kernel (2) of [news] 三: keys as block-wise per-channel INT2
 * (each channel's step and zero shared by c->key_group consecutive tokens:
 * 32, or the larger groups 64 and 128 that [rainbus] 局限与改进 (1) names as
 * untested; every 32-token record of a group carries the group's step and
 * zero), values as per-token INT2 ([rainbus] 方法步骤详情 (2)(3)).  Per
 * group: zero = min,
 * step = (max - min)/3 in fp32, code = round-half-even((x - zero)/step)
 * clamped to [0,3] (0 when max == min); step and zero stored as fp16.
 * Tokens [0, n_tok) of each (b,h) row of the sources are written to packed
 * positions [n_packed, n_packed + n_tok); then c->n_packed += n_tok.
 *  k_hat  bf16 [B][Hkv][src_T][128] rotated, scaled keys (from oscar_rotate_scale_k)
 *  k_norm fp16 [B][Hkv][src_T]      their norms
 *  v      bf16 [B][Hkv][src_T][128] values
 * Flush mode: k_hat == k_norm == v == NULL quantises the full residual window
 * (requires c->n_res == 128, src_T and n_tok ignored) and sets c->n_res = 0
 * ([news] 三: batch quantisation once 128 tokens have accumulated).
 * Requires n_tok a multiple of the key group, src_T >= n_tok, c->n_res == 0 in
 * non-flush mode (packed tokens precede residual ones) and
 * c->n_packed + n_tok <= c->T_cap (else OSCAR_ERR_CAPACITY).
 */
oscar_status oscar_quantize_kv(oscar_cache* c, const oscar_bf16* k_hat, const oscar_f16* k_norm,
                               const oscar_bf16* v, int src_T, int n_tok, void* stream);

/*
 * Fused prefill: kernels (1) and (2) of [news] 三 in one pass over a prefix.
 * Each key is rotated and scaled exactly as oscar_rotate_scale_k does (same
 * k_hat bits, same norm), then keys and values are quantised and packed
 * exactly as oscar_quantize_kv does, without k_hat or a value copy ever
 * going through global memory (598 B of HBM traffic per token-head instead
 * of the ~1.6 KB of the two-call path).  Tokens [0, n_tok) of each (b,h) row
 * are written to packed positions [n_packed, n_packed + n_tok); then
 * c->n_packed += n_tok; the rotation and scaling flags are c->flags.
 *  k  bf16 [B][Hkv][in_T][128] raw keys (row stride in_T tokens)
 *  v  bf16 [B][Hkv][in_T][128] values
 * Requires n_tok a multiple of the key group, in_T >= n_tok, c->n_res == 0 and
 * c->n_packed + n_tok <= c->T_cap (else OSCAR_ERR_CAPACITY); pointers
 * 16-byte aligned.
 */
oscar_status oscar_prefill_kv(oscar_cache* c, const oscar_bf16* k, const oscar_bf16* v, int in_T,
                              int n_tok, void* stream);

/*
 * Cache update for n_tok new tokens per (b,h) row, one after another: before
 * each token, a full residual window (128 tokens) is flushed as in
 * oscar_quantize_kv flush mode; the token's key is rotated and scaled into
 * residual slot n_res, its value copied next to it, and c->n_res grows
 * (flush-before-append: the newest token always stays 16-bit).  A decode
 * step calls it with n_tok = 1.  ([notes] End-to-End Flow; [news] 三.)
 *  k_new, v_new  bf16 [B][Hkv][n_tok][128] raw keys and values
 * Fails with OSCAR_ERR_CAPACITY, launching nothing, if the flushes the call
 * needs do not fit in T_cap.
 */
oscar_status oscar_append_kv(oscar_cache* c, const oscar_bf16* k_new, const oscar_bf16* v_new,
                             int n_tok, void* stream);

/*
 * Fused dequantisation + inverse token scaling + attention (kernel (3) of
 * [news] 三; [notes] End-to-End Flow: "Q.K^T and dequantization fused into a
 * single kernel", III Efficiency), split-K over tokens (flash-decoding) with
 * a log-sum-exp combine.  For query head j of sequence b, with h = j / g:
 *   score_t = softmax_scale * q'_j . k_t,   k_t = (c*step + zero) * norm (packed)
 *                                           k_t = k_hat_t * norm_t       (residual)
 *   out_j   = sum_t softmax(score)_t * v_t, v_t = c*step + zero (packed) or v_res_t
 * over the c->n_packed packed and c->n_res residual tokens of row (b, h).
 * The records are read as the cache's fields say: INT2 or INT4 codes
 * (c->bits), each 32-token record with its key group's step and zero
 * (c->key_group), norms stored as n / target (c->norm_target; the product
 * with k_hat is the same key), per-head or all-heads norms (c->flags).
 *  q_rot      fp32 [B][Hq][128] rotated queries (oscar_rotate_q)
 *  out        fp32 [B][Hq][128]; an empty cache gives zeros
 *  num_splits packed-token splits per (b,h); 0 = choose for this device
 *             (oscar_decode_num_splits); one more split handles the residual.
 *  workspace  device scratch of at least oscar_decode_workspace_bytes(B, Hkv,
 *             Hq, n_packed, splits) bytes (16-byte aligned), caller-owned.
 *             Layout: a header of OSCAR_DECODE_WS_HEADER_BYTES (one 32-bit
 *             arrival counter for each of up to 65536 (b, h) rows), then the
 *             split-K partial records, B*Hq*(splits+1) records of 528 bytes.
 *             The row's last CTA to finish combines the row's partials (no
 *             second kernel is launched) and sets its counter back to zero.
 *             So the header must be zero before a workspace's first use
 *             (cudaMemset it once after allocating); every call leaves it
 *             zero, whatever its shape or split count, and the rest needs no
 *             initialisation.  A counter found non-zero is reported in the
 *             device status word (oscar_device_status) and that row's output
 *             is not written.  B*Hkv must not exceed 65536 (B*Hkv*2 for
 *             groups of 9 to 16 query heads, which take two rows per KV head;
 *             else OSCAR_ERR_UNSUPPORTED).  Calls that use one workspace must
 *             not overlap on the GPU.
 */
oscar_status oscar_decode_attention(const oscar_cache* c, const float* q_rot, int Hq,
                                    float softmax_scale, float* out, int num_splits,
                                    void* workspace, size_t ws_bytes, void* stream);

/*
 * Fused decode step: oscar_rotate_q, oscar_append_kv of one token and
 * oscar_decode_attention in one kernel launch (plus the flush of a full
 * residual window, before it, as oscar_append_kv does).  The kernel's CTAs
 * rotate their own query heads, and the residual CTA of each (b, h) row
 * rotates and scales the new key, writes it and the new value at the next
 * residual slot, then attends over the window including it; the other CTAs
 * never read the window.  The rotation and scaling are the same device code
 * as in the separate calls, so the outputs and the cache equal theirs bit
 * for bit ([news] 三: kernels ① and ③ around one decode step; [notes] II
 * End-to-End Flow).
 *  q          bf16 [B][Hq][128] raw queries
 *  k_new      bf16 [B][Hkv][128] raw key of the new token
 *  v_new      bf16 [B][Hkv][128] value of the new token
 *  out, num_splits, workspace: as for oscar_decode_attention, the split count
 *             planned for n_packed after the flush (if any).
 * Contiguous caches only (a paged cache uses the oscar_paged_* calls).  All
 * checks, including capacity for the flush and the workspace size, happen
 * before any launch; n_res (and n_packed after a flush) advance on success.
 * If the flush launched and the decode launch then fails, the flush stays.
 */
oscar_status oscar_decode_step(oscar_cache* c, const oscar_bf16* q, const oscar_bf16* k_new,
                               const oscar_bf16* v_new, int Hq, float softmax_scale, float* out,
                               int num_splits, void* workspace, size_t ws_bytes, void* stream);

/* Split count oscar_decode_attention uses for num_splits = 0 on the current
 * device (>= 1).  Returns 1 when no device can be queried. */
int oscar_decode_num_splits(int B, int Hkv, int Hq, int n_packed);

/* The planner behind oscar_decode_num_splits, for a device of `sms`
 * multiprocessors that hold `ctas_per_sm` decode CTAs each: rows = B*Hkv,
 * n_blocks = n_packed / 32.  Host arithmetic only (no CUDA call); returns a
 * count in [1, 512], 1 for non-positive arguments. */
int oscar_decode_plan_splits(long long rows, long long n_blocks, int ctas_per_sm, int sms);

/* Workspace bytes needed by oscar_decode_attention / oscar_paged_decode_attention
 * (and enough for oscar_bf16_decode_attention) for `num_splits` token splits
 * (0 = the automatic count for n_packed tokens): the counter header plus
 * B*Hq*(splits+1)*528 bytes of partial records. */
#define OSCAR_DECODE_WS_HEADER_BYTES (65536u * 4u)
size_t oscar_decode_workspace_bytes(int B, int Hkv, int Hq, int n_packed, int num_splits);

/*
 * Comparison kernel: unquantised bf16 split-K flash-decoding attention with
 * the same grid, split and combine scheme (the "BF16 FlashDecoding-v2"
 * baseline of [notes] III Efficiency).  No rotation, no scaling.
 *  q      bf16 [B][Hq][128]
 *  K, V   bf16 [B][Hkv][T_stride][128], tokens [0, T) of each row used
 *  out    fp32 [B][Hq][128]
 *  workspace as for oscar_decode_attention (use n_packed = T for sizing).
 */
oscar_status oscar_bf16_decode_attention(const oscar_bf16* q, const oscar_bf16* K,
                                         const oscar_bf16* V, int B, int Hq, int Hkv, int T,
                                         int T_stride, float softmax_scale, float* out,
                                         int num_splits, void* workspace, size_t ws_bytes,
                                         void* stream);

/* Size of the static device array behind oscar_decode_attention_static_ws. */
#define OSCAR_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * oscar_decode_attention without a workspace argument, for callers that
 * cannot allocate device memory: for example a serving loop that allows no
 * cudaMalloc after start-up (it can stall the device and fragment memory),
 * or a plug-in whose host runtime owns all device memory and lends it no
 * allocator.  The pages have no counterpart: this is an integration aid.
 * Same arguments, results and checks as oscar_decode_attention, except that
 * the split-K partial records and the row counters (the workspace of
 * oscar_decode_attention) live in a 16 MiB array inside the library
 * (OSCAR_STATIC_SCRATCH_BYTES), which every GPU that loads the library keeps
 * until the process exits.  The call allocates nothing.
 *  - The workspace, oscar_decode_workspace_bytes(B, Hkv, Hq, n_packed,
 *    splits), must fit in that array.  With num_splits = 0 the automatic
 *    split count is lowered to the largest that fits (at least 1); an
 *    explicit count that does not fit, or a batch whose single split does
 *    not fit, returns OSCAR_ERR_WORKSPACE and launches nothing.  For
 *    example a batch-48, 32-query-head, 8-KV-head layer at the 11 splits
 *    the planner gives a 128K context needs 256 KiB + 48*32*12*528 bytes,
 *    about 10.0 MB.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress); make it before any stream
 *    capture.  A failed lookup returns OSCAR_ERR_CUDA.
 *  - Every call shares the one array and it keeps the last call's contents;
 *    calls whose kernels overlap on the GPU (e.g. on two streams) race on it.
 *    Its counter header starts zeroed when the library loads and every call
 *    leaves it zero; each call writes every partial record it reads.
 */
oscar_status oscar_decode_attention_static_ws(const oscar_cache* c, const float* q_rot, int Hq,
                                              float softmax_scale, float* out, int num_splits,
                                              void* stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * word.  OSCAR_OK if no kernel recorded an error, else OSCAR_ERR_DEVICE_STATUS. */
oscar_status oscar_device_status(void* stream);

/*
 * Paged cache calls (oscar_paged_cache).  Each does, per sequence, what the
 * contiguous call of the same name does for the whole batch; lengths are
 * read from and written to the device arrays by the kernels.
 *
 * oscar_paged_prefill_kv: the fused prefill of raw keys and values
 * k, v bf16 [B][Hkv][in_T][128]: sequence b's tokens [0, n_tok[b]) are
 * rotated, scaled, quantised and written to its logical blocks
 * n_packed[b]/32 .. onwards; then n_packed[b] += n_tok[b].  n_tok: device
 * int32 [B], each a multiple of the key group and <= max_tok (a host bound sizing the
 * launch, <= in_T); requires n_res[b] == 0 for sequences with n_tok[b] > 0.
 *
 * oscar_paged_append_kv: one new token (k_new, v_new bf16 [B][Hkv][128])
 * for every sequence b with active[b] != 0 (active NULL: all): a full
 * residual window is flushed first into the sequence's next 4 logical
 * blocks, then the token is rotated, scaled and stored at residual slot
 * n_res[b] (flush-before-append, as oscar_append_kv).
 *
 * oscar_paged_decode_attention: oscar_decode_attention over every
 * sequence's own n_packed[b] + n_res[b] tokens.  max_packed (host) bounds
 * the n_packed[b] and plans the splits (num_splits 0: planned from it):
 * with c = ceil(max_packed / 32 / splits) blocks, sequence b's n_packed[b]/32
 * blocks are cut into ceil(n/c) splits of equal length (at most `splits`; a
 * sequence longer than max_packed spreads over all of them), so a shorter
 * sequence fills fewer splits.  The workspace is
 * oscar_decode_workspace_bytes(B, Hkv, Hq, max_packed, splits).
 * A sequence with no tokens gives zeros.
 *
 * The device-side checks of a page id outside [0, n_pages) or a length
 * outside its range skip the access and record an error in the status word
 * (oscar_device_status).
 */
oscar_status oscar_paged_prefill_kv(oscar_paged_cache* c, const oscar_bf16* k,
                                    const oscar_bf16* v, int in_T, const int32_t* n_tok,
                                    int max_tok, void* stream);
oscar_status oscar_paged_append_kv(oscar_paged_cache* c, const oscar_bf16* k_new,
                                   const oscar_bf16* v_new, const int32_t* active, void* stream);
oscar_status oscar_paged_decode_attention(const oscar_paged_cache* c, const float* q_rot, int Hq,
                                          float softmax_scale, int max_packed, float* out,
                                          int num_splits, void* workspace, size_t ws_bytes,
                                          void* stream);

/* Self-test of the bounded waits (failure detection; the pages have no
 * counterpart).  One CTA waits on an mbarrier that nothing arrives at,
 * gives up after `iterations` polls, records the wait-timeout bit in the
 * device status word exactly as a decode whose copies never landed would,
 * and returns: no fault, no hang, the context stays usable.  Afterwards
 * oscar_device_status reports OSCAR_ERR_DEVICE_STATUS (and clears the word).
 * iterations: 1 .. 1<<20, else OSCAR_ERR_INVALID_ARG (nothing launched). */
oscar_status oscar_selftest_wait_timeout(unsigned iterations, void* stream);

/* Static description of a status code. */
const char* oscar_status_string(oscar_status s);

/* Number of kernels this library has launched in this process. */
unsigned long long oscar_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
