/*
 * kvq.h -- C ABI of the quantized KV-cache library for NVIDIA B300 (sm_103a).
 *
 * Two hot-path calls and one host utility:
 *
 *   kvq_append       quantize-on-append: block-diagonal Walsh-Hadamard rotation
 *                    of each new K/V head vector, token-wise asymmetric INT-b
 *                    quantization with one fp16 scale and zero per (token, head),
 *                    packed into a paged cache; optional bf16 recent-token window.
 *   kvq_decode_attn  split-K decode attention that reads the packed codes,
 *                    dequantizes in registers and scores them against the
 *                    once-rotated query; merges the bf16 window; writes fp32 o.
 *   kvq_alloc_bits   RateQuant greedy marginal-gain allocation of per-component
 *                    bit-widths (host only).
 *   kvq_distortion   per-head quantization MSE at several widths (calibration),
 *   kvq_fit_distortion  and the (alpha, beta) fit of D(b) = alpha beta^-b.
 *
 * Conventions shared by every call
 *   - Every pointer marked "device" is caller-owned device memory (e.g. from
 *     PyTorch).  The library allocates no memory and never synchronises a
 *     stream; kernels are launched on the stream passed in (NULL = legacy
 *     default stream).
 *   - Arguments that can be checked on the host are checked before any launch;
 *     a failed check returns KVQ_EINVAL / KVQ_EUNSUPPORTED and launches nothing.
 *     kvq_last_error() then holds a message (thread-local).
 *   - Errors that only the device can see (a page id outside [0, num_pages), a
 *     sequence longer than its page-table row, a vector whose scale or zero is
 *     not finite in fp16, an asynchronous copy that did not complete in time)
 *     are OR-ed into the cache's device status word; the affected work is
 *     skipped, nothing traps.  Read it with kvq_get_status() after
 *     synchronising the stream.
 *   - Position p of sequence b lives in logical page p / 16, slot p % 16;
 *     page_table[b * max_pages + p / 16] names the physical page.
 *
 * Page layout (layer l; a convention of this library -- the pages only say that
 * a paged-attention server stores the cache in uniform blocks):
 *   for each KV head h = 0 .. Hkv-1, a contiguous 16-byte-aligned segment
 *     K codes  [16][head_dim * bK / 8]   token-major
 *     V codes  [16][head_dim * bV / 8]
 *     K (s, z) [16] x {fp16 s, fp16 z}
 *     V (s, z) [16] x {fp16 s, fp16 z}
 *   codes packed little-endian: element j at bit (j * b) % 8 of byte (j * b) / 8.
 *   page_bytes(l) = sum_h 16 * (head_dim * (bK_h + bV_h) / 8 + 8).
 *
 * Rotation and quantizer (what a stored vector means)
 *   u = H_blk x, H_blk = diag(H_n, ..., H_n), H_n the Sylvester Hadamard matrix
 *   (entries (-1)^popcount(i & j), unnormalised).  Per (token, head, K|V):
 *     z = fp16_round_down(min u),  s = fp16_round_up((max u - z) / (2^b - 1)),
 *     c_j = round_half_even((u_j - z) * (1 / s)),   deq_j = c_j * s + z,
 *   with u, u - z and 1 / s rounded to fp32.  Since H_n H_n = n I,
 *   q . k = (H q) . (H k) / n and x = H u / n.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_EINVAL = 1,        /* bad argument (null pointer, bad size, misalignment) */
  KVQ_EUNSUPPORTED = 2,  /* valid but not built: head_dim, block, bits, GQA group */
  KVQ_ECUDA = 3,         /* a CUDA runtime call failed (message in kvq_last_error) */
  KVQ_EBUDGET = 4,       /* kvq_alloc_bits: budget below the minimum allocation */
  KVQ_EDEVICE = 5,       /* kvq_get_status: the device status word is non-zero */
  KVQ_EWORKSPACE = 6     /* kvq_decode_attn: workspace smaller than required */
} kvq_status;

/* Bits of the device status word (OR-ed together by kernels). */
#define KVQ_DEV_BAD_PAGE      0x1  /* page id outside [0, num_pages) */
#define KVQ_DEV_BAD_LENGTH    0x2  /* seq_len < 0 or beyond max_pages * 16 */
#define KVQ_DEV_NONFINITE     0x4  /* scale or zero not finite in fp16 (input out of range) */
#define KVQ_DEV_COPY_TIMEOUT  0x8  /* an asynchronous page copy did not complete in time */

/* Descriptor of a paged quantized cache.  Plain data; the library keeps no
 * reference to it after a call returns. */
typedef struct kvq_cache {
  int num_layers;
  int num_kv_heads;          /* Hkv, 1 .. 64 */
  int head_dim;              /* d: 64 or 128 */
  int page_size;             /* must be 16 */
  int had_block;             /* Hadamard block n: 32, 64 or 128, dividing head_dim;
                                1 = no rotation (u = x), the plain token-wise quantizer
                                that the SAW-INT4 page contrasts with the rotated one */
  int window;                /* R: bf16 recent-token window (0 = none), 0 .. 1024 */
  int max_batch;             /* sequences addressable in each window buffer */
  int num_pages;             /* physical pages in each layer pool */
  const int8_t* bits_host;   /* host [num_layers][num_kv_heads][2] (bK, bV), each 2, 4 or 8 */
  void* const* layer_pools;  /* host array [num_layers] of device pointers, each
                                num_pages * kvq_page_bytes(layer) bytes, 16-byte aligned */
  void* const* window_bufs;  /* host array [num_layers] of device pointers to bf16
                                [max_batch][Hkv][2][R][head_dim] (window R > 0), to the
                                LogQuant reserve [max_batch][Hkv][2][kvq_logquant_rows(W)]
                                [head_dim] (logquant_w = W > 0), or to the key-per-channel
                                ring [max_batch][Hkv][2][R + 16][head_dim] (key_per_channel,
                                any R), kvq_window_bytes() bytes each; NULL when none of
                                them is used.  Sequence b of a call
                                uses row b; a call for a subset of a batch (e.g. a
                                one-sequence prefill) passes a descriptor whose pointers
                                are offset to its rows. */
  int* status_dev;           /* device int, the sticky status word (may be NULL) */
  int launch_flags;          /* 0 or KVQ_LAUNCH_OVERLAP (decode calls only) */
  int logquant_w;            /* 0, or W: LogQuant log-spaced full-precision tokens with
                                base window W, a power of two in [2, 256]; needs window 0 */
  int key_per_channel;       /* 0, or 1: keys quantized symmetrically per channel, one fp16
                                scale per (page, KV head, channel) (see below); not with
                                logquant_w */
} kvq_cache;

/*
 * Key-per-channel mode (key_per_channel = 1).  Follows the RateQuant technical
 * summary, Methodology section 3 (KIVI quantizes keys symmetrically per channel
 * and values asymmetrically per token) and "LogQuant ...", section 5 (2-bit
 * quantization with a key-per-channel strategy).  The 16 keys of a page form a
 * group (a reading: the pages give no group size): after the rotation,
 *   s_j = fp16_round_up(max_t |u_tj| / Q),  Q = 2^(bK-1) - 1,
 *   c_tj = round_half_even(u_tj * (1 / s_j))  in [-Q, Q],   deq_tj = c_tj * s_j,
 * with max |u| / Q and 1 / s rounded to fp32; s_j = 0 gives c = 0.  Values keep
 * the token-wise rule.  A page is quantized once all of its positions have left
 * the window: with length L, positions 0 .. Q(L) - 1 are quantized, Q(L) =
 * 16 floor(max(L - R, 0) / 16), and positions Q(L) .. L - 1 (at most R + 15)
 * keep bf16 K and V in a ring of R + 16 rows, slot p % (R + 16), so the mode
 * needs window_bufs even with R = 0.  Page segment of head h:
 *   K codes  [16][head_dim * bK / 8]   stored c + 2^(bK-1), packed as above
 *   V codes  [16][head_dim * bV / 8]
 *   K scales [head_dim] x fp16
 *   V (s, z) [16] x {fp16 s, fp16 z}
 * page_bytes(l) = sum_h (16 * head_dim * (bK_h + bV_h) / 8 + 2 * head_dim + 64).
 * kvq_append quantizes the pages the append completes, then writes the new bf16
 * rows (two launches); kvq_decode_step runs the append of its token and then
 * the decode (two launches).
 */

/*
 * LogQuant mode (logquant_w = W > 0).  Follows "LogQuant: Log-Distributed
 * 2-Bit Quantization of KV Cache with Superior Accuracy Preservation",
 * Methodology section 2 (base window W, the newest tokens at full precision,
 * older ones selected ever more sparsely, a 3W full-precision reserve whose
 * older selections are halved as it fills) and section 4 (A V = A_P V_P).
 * Every token is quantized into its page on arrival, as without a window.
 * Besides, a set B of positions keeps its bf16 K and V in the reserve: every
 * new token joins B; when |B| reaches 3W, of the oldest 2W members (by
 * position) every other one stays, the first of each pair.  Decode attention
 * uses the bf16 values for the members of B and the quantized ones for every
 * other token.  B depends on the length alone (kvq_logquant_members lists it).
 */

/* Rows of one (sequence, KV head, K|V) plane of the LogQuant reserve for base
 * window W: 3W ring rows and log2(W) + 1 level buffers of W / 2 rows; 0 when W
 * is not a power of two in [2, 256]. */
int kvq_logquant_rows(int w);

/* The positions of B after n appends with base window W (host only), ascending,
 * into positions[0 .. max) when positions is not NULL; returns |B|, or -1 when
 * W is not a power of two in [2, 256] or n < 0. */
long long kvq_logquant_members(long long n, int w, long long* positions, long long max);

/* Bytes of window_bufs[layer] this descriptor needs (the bf16 window, the
 * LogQuant reserve or the key-per-channel ring, for max_batch sequences); 0 when
 * it needs none or on a bad descriptor. */
size_t kvq_window_bytes(const kvq_cache* cache);

/*
 * KVQ_LAUNCH_OVERLAP: decode launches (kvq_decode_attn, kvq_decode_attn_static,
 * kvq_decode_step) use programmatic dependent launch.  The kernel may start
 * while the kernel launched just before it on the stream is still running.  Before
 * that kernel has completed, it reads only the page table, the sequence lengths
 * and the layer's pool, and it starts the page copies.  It waits for that
 * kernel's completion before reading q, K_new, V_new or the window, and before
 * writing anything.  Contract: the preceding kernel does not write this layer's
 * pool, the page table or seq_lens.  A preceding kvq_decode_step of the same layer
 * writes that pool, for example.  A copy or memset in between orders the
 * launches as usual.
 */
#define KVQ_LAUNCH_OVERLAP 0x1

/* Bytes of one page of `layer` (layout above); 0 on a bad descriptor. */
size_t kvq_page_bytes(const kvq_cache* cache, int layer);

/*
 * kvq_append -- quantize-on-append.
 * Follows "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization for Real-World LLM
 * Serving" (summary; section 2, block-diagonal Hadamard rotation before
 * quantization; section 3, the fused engine doing rotation and quantization in
 * the same memory pass) and the RateQuant technical summary, Methodology
 * section 3 (K and V as separate components with their own bit-widths, taken
 * here from cache->bits_host).  The recent-token window follows "LogQuant:
 * Log-Distributed 2-Bit Quantization of KV Cache ...", Methodology section 2
 * (most recent tokens kept at full precision).
 *
 *   K, V        device bf16 [B][T_new][Hkv][head_dim], contiguous, 16-byte aligned.
 *   page_table  device int32 [B][max_pages]; must cover every position written.
 *   seq_lens    device int32 [B]: tokens already in each sequence BEFORE this call
 *               (window included); they are not modified.
 * Appended token i of sequence b takes position p = seq_lens[b] + i.  With R = 0
 * it is quantized into its page slot.  With R > 0, positions p < L - R (L the new
 * length) are quantized -- tokens leaving the window are read from the ring slot
 * p % R of window_bufs[layer] before it is overwritten -- and the last min(L, R)
 * positions are copied to the ring.  In LogQuant mode every token is quantized,
 * and the members of B after the append get their bf16 rows in the reserve
 * (one more launch first moves the older members that this append's halvings
 * thin out of the reserve's ring).  In the key-per-channel mode a page is
 * quantized when the append completes it and all of its positions have left
 * the window (rows of older positions come from the ring), and the appended
 * positions from max(seq_lens[b], Q(L)) on are copied to the ring (a second
 * launch).  Two appends to one sequence must be stream-ordered.  Returns
 * KVQ_OK once the kernels are enqueued.
 */
kvq_status kvq_append(const kvq_cache* cache, int layer, const void* K, const void* V,
                      const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                      int B, int T_new, void* stream);

/* Workspace bytes kvq_decode_attn needs for this (B, Hq, max_pages) on the
 * current device; 0 on a bad argument.  The workspace must be zero-filled once
 * before its first use (e.g. torch.zeros); every call leaves it ready for the
 * next.  Two calls that run concurrently must not share a workspace. */
size_t kvq_decode_workspace_bytes(const kvq_cache* cache, int B, int Hq, int max_pages);

/*
 * kvq_decode_attn -- one decode step of attention over the quantized cache.
 * Follows "SAW-INT4 ..." section 3 (attention consumes the compact cache, the
 * rotation undone on the fly: the query is rotated once, q . k = (H q).(H k)/n),
 * "LogQuant ..." Methodology section 4 (attention is independent of the order of
 * the (key, value) pairs, A V = A_P V_P, so split-K partials, quantized pages
 * and the bf16 window may be combined in any order) and Methodology section 2
 * (full-precision recent window).
 *
 *   q            device [B][Hq][head_dim], bf16 (q_is_fp32 = 0) or fp32 (1).
 *                Query head h reads KV head h / (Hq / Hkv); Hq / Hkv in {1, 2, 4}.
 *   seq_lens     device int32 [B]: tokens per sequence INCLUDING the window.
 *   softmax_scale  multiplies q . k; pass 0 for 1 / sqrt(head_dim).
 *   o            device fp32 [B][Hq][head_dim], written.  A sequence of length 0
 *                gets o = 0.
 *   workspace    device, ws_bytes >= kvq_decode_workspace_bytes(cache, B, Hq,
 *                max_pages), 16-byte aligned, zero-filled before its first use.
 * In LogQuant mode the quantized splits leave out the members of B, and one to
 * four more CTAs per (sequence, KV head) attend over their bf16 rows in the
 * reserve (more of them when the batch leaves the wave room).  In
 * the key-per-channel mode the splits read each page's channel scales and one
 * more CTA attends over the ring's positions Q(L) .. L - 1.
 * One kernel launch.  Returns KVQ_OK once enqueued.
 */
kvq_status kvq_decode_attn(const kvq_cache* cache, int layer, const void* q, int q_is_fp32,
                           const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                           int B, int Hq, float softmax_scale, float* o, void* workspace,
                           size_t ws_bytes, void* stream);

/*
 * kvq_decode_step -- one decode step with the new token fused in: the same
 * result, in the cache and in o, as kvq_append of one token per sequence
 * followed by kvq_decode_attn, in a single launch.
 * Follows "SAW-INT4 ..." section 3 (the fused engine: rotation and
 * quantization of the newest token happen inside the same memory pass as the
 * attention that reads the compact cache) and "LogQuant ..." Methodology
 * section 2 (the newest token enters the full-precision window).
 *
 *   K_new, V_new device bf16 [B][Hkv][head_dim], 16-byte aligned: this step's
 *                token of every sequence.
 *   seq_lens     device int32 [B]: tokens per sequence INCLUDING this step's
 *                token (>= 1; a length below 1 sets KVQ_DEV_BAD_LENGTH and
 *                the sequence is skipped).
 *   Every other argument as for kvq_decode_attn.
 * Position len - 1 of sequence b takes the new token.  Without a window it is
 * quantized into its page slot; with R > 0 it enters ring slot (len - 1) % R,
 * and the token it replaces (position len - 1 - R, if any) is quantized into
 * its page slot.  In LogQuant mode it is quantized into its page slot and its
 * bf16 rows enter the reserve; when this token fills B to 3W, the halving's
 * block moves from the reserve's ring to its level buffer in the same launch.
 * In the key-per-channel mode the step is kvq_append of the token (whose page,
 * once complete and out of the window, is quantized) followed by the decode:
 * three launches.  Two steps on one cache must be stream-ordered.  Otherwise
 * one kernel launch.  Returns KVQ_OK once enqueued.
 */
kvq_status kvq_decode_step(const kvq_cache* cache, int layer, const void* K_new,
                           const void* V_new, const void* q, int q_is_fp32,
                           const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                           int B, int Hq, float softmax_scale, float* o, void* workspace,
                           size_t ws_bytes, void* stream);

/*
 * kvq_decode_attn_static -- kvq_decode_attn without a caller workspace.
 * The pages have no counterpart of this call: it exists for callers that cannot
 * allocate device memory -- a plugin inside a host process whose device memory
 * is owned and budgeted by that process's allocator, or a latency-critical path
 * that must not reach cudaMalloc / cudaFree because they can synchronise the
 * device.  It runs the same decode as kvq_decode_attn (same arguments minus
 * workspace and ws_bytes) with its scratch in a fixed device array of
 * KVQ_STATIC_WORKSPACE_BYTES owned by the library, which every GPU that loads
 * the library holds until the process exits.  It calls no allocating routine.
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress; the first such query on a device loads the
 *     module there), so make the first call on a device before any stream
 *     capture.  Looking it up each time keeps the call correct after a device
 *     reset.
 *   - Every call shares the array and it keeps the last call's contents; the
 *     call clears the part that must start at zero (an async memset on
 *     `stream`) itself.  That memset also orders the decode after the previous
 *     kernel on the stream, so KVQ_LAUNCH_OVERLAP has no effect here.  Calls
 *     whose work overlaps on the GPU (other streams, other host threads) race
 *     on the array: serialise them.
 *   - Returns KVQ_EWORKSPACE, launching nothing, when the decode needs more
 *     scratch than KVQ_STATIC_WORKSPACE_BYTES (kvq_decode_workspace_bytes tells
 *     how much); use kvq_decode_attn with a workspace then.
 */
#define KVQ_STATIC_WORKSPACE_BYTES (8 * 1024 * 1024)
kvq_status kvq_decode_attn_static(const kvq_cache* cache, int layer, const void* q,
                                  int q_is_fp32, const int32_t* page_table, int max_pages,
                                  const int32_t* seq_lens, int B, int Hq, float softmax_scale,
                                  float* o, void* stream);

/*
 * kvq_alloc_bits -- RateQuant greedy marginal-gain bit allocation (host only).
 * Follows the RateQuant technical summary, Methodology section 1 (distortion
 * model D(b) = alpha * beta^-b, objective min sum_i w_i D_i(b_i) subject to
 * sum_i b_i = B) and section 3 (integer refinement by a greedy marginal-gain
 * loop; K and V as 2N independent components with their own beta).
 *
 *   w[n]          sensitivities with alpha folded in, > 0.
 *   beta[n]       distortion decay rates, > 1.
 *   budget        total bits sum_i b_i may not exceed.
 *   allowed_mask  [n] (or NULL = {2, 4, 8} for all): bit b set means width b
 *                 (1 .. 15) is allowed for component i.
 *   bits_out[n]   written; leftover (may be NULL) receives budget - sum(bits).
 * Every component starts at its smallest allowed width; while a step fits the
 * remaining budget, the step to the next allowed width with the largest gain per
 * bit w_i (beta_i^-b - beta_i^-b') / (b' - b) is taken (ties: lowest index).
 * Returns KVQ_EBUDGET (bits_out untouched) if the budget is below the minimum.
 * Component order for a cache: (layer * Hkv + head) * 2 + kv, kv = 0 for K.
 */
kvq_status kvq_alloc_bits(const double* w, const double* beta, int n, long long budget,
                          const uint16_t* allowed_mask, int* bits_out, long long* leftover);

/*
 * kvq_distortion -- distortion calibration: the mean-squared error of this
 * library's quantizer (rotation, fp16 scale and zero, round-half-even codes,
 * as stored by kvq_append) at several bit-widths, per KV head, on a sample of
 * K or V vectors.  Follows the RateQuant technical summary, Methodology
 * section 3 (fit the distortion model D(b) = alpha * beta^-b of the quantizer
 * actually used, on a small calibration set, per K and V component) and
 * section 4 (the fit takes 5 bit-widths).
 *
 *   head_dim, had_block  as in kvq_cache (64 | 128; 1 | 32 | 64 | 128 dividing it).
 *   X        device bf16 [T][num_kv_heads][head_dim], 16-byte aligned: T vectors
 *            per head (e.g. a batch of calibration sequences, flattened).
 *   widths   host int [n_widths], each 1 .. 8; n_widths 1 .. 8.
 *   mse      device double [num_kv_heads][n_widths], 8-byte aligned, overwritten
 *            with sum over the T vectors of |x - deq(x)|^2 / (T * head_dim) in the
 *            model's basis.  The orthonormal rotation keeps that norm, so it is
 *            sum |u - deq(u)|^2 / (had_block * T * head_dim), where u is the
 *            unnormalised rotation.
 * A width-b code is c = round-half-even((u - z) / s) with M = 2^b - 1 levels, as
 * for the cache's 2-, 4- and 8-bit codes.  Zeroes mse and launches one kernel on
 * `stream`.  Per-CTA sums are added in fp64 atomically, so the last bits depend
 * on their order.  T == 0 gives zeros.
 */
kvq_status kvq_distortion(int head_dim, int had_block, int num_kv_heads, const void* X,
                          long long T, const int* widths, int n_widths, double* mse,
                          void* stream);

/*
 * kvq_fit_distortion -- least-squares fit of ln D(b) = ln alpha - b ln beta per
 * component (host only), the distortion model of the RateQuant technical
 * summary, Methodology section 1, fitted as in section 3.
 *
 *   mse    host double [n][n_widths] (e.g. kvq_distortion's output, copied back).
 *   widths host int [n_widths], distinct.
 *   alpha, beta  host double [n], written.
 * Widths whose D is not positive and finite (a lossless width) are left out.  A
 * component with fewer than two widths left takes beta = 4: one more bit halves a
 * uniform quantizer's step and quarters its error.  Its alpha then comes from the
 * width left (D(b) 4^b), or is 0 when none is left.  The result feeds
 * kvq_alloc_bits as w_i = sensitivity_i * alpha_i, beta_i.
 */
kvq_status kvq_fit_distortion(const double* mse, const int* widths, int n_widths, int n,
                              double* alpha, double* beta);

/* Copy the device status word into *device_status (synchronous copy; the caller
 * synchronises the streams that ran kernels first).  Returns KVQ_EDEVICE when it
 * is non-zero, KVQ_OK when it is zero. */
kvq_status kvq_get_status(const kvq_cache* cache, int* device_status);

/* Zero the device status word on `stream`. */
kvq_status kvq_reset_status(const kvq_cache* cache, void* stream);

/* Message of the last failed call on this thread ("" if none). */
const char* kvq_last_error(void);

/* Library version string, e.g. "kvq 0.1 sm_103a". */
const char* kvq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H_ */
