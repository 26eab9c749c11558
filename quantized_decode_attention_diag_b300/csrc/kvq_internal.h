// Internal interface between the C ABI (kvq_api.cpp) and the kernels.
// Plain structs passed by value as kernel parameters (well under 4 KB).
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int kPage = 16;        // tokens per page (= MMA M dimension)
constexpr int kMaxHeads = 64;    // KV heads per layer
constexpr int kMaxWindow = 1024; // bf16 recent-token window
constexpr int kMaxGroup = 4;     // query heads per KV head handled per CTA

// Division by a divisor fixed for a launch, for 0 <= n < 2^31 and 1 <= d < 2^31:
// floor(n / d) = (mulhi(m, n) + n) >> l with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1 (T. Granlund and P. L. Montgomery, "Division
// by invariant integers using multiplication", PLDI 1994, section 4).  Then
// 2^(32+l) < (2^32 + m) d <= 2^(32+l) + 2^l, which makes the quotient exact, and
// mulhi(m, n) < n keeps the sum below 2^32.
struct FastDiv {
  uint32_t m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.l = 0;
  while ((1ull << f.l) < d) ++f.l;
  f.m = static_cast<uint32_t>((((1ull << f.l) - d) << 32) / d + 1);
  return f;
}
__host__ __device__ inline uint32_t fastdiv(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
  const uint32_t hi = __umulhi(n, f.m);
#else
  const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(n) * f.m) >> 32);
#endif
  return (hi + n) >> f.l;
}

// Per-layer page geometry, computed on the host from the bits table.
struct LayerGeom {
  int head_off[kMaxHeads];       // byte offset of head h's segment in a page
  int8_t bits[kMaxHeads][2];     // (bK, bV)
  long long page_bytes;
  int max_head_bytes;            // largest head segment (one async copy)
};

struct AppendParams {
  const uint16_t* K;             // bf16 [B][T][Hkv][D]
  const uint16_t* V;
  uint8_t* pool;                 // [num_pages][page_bytes]
  uint16_t* window;              // bf16 [max_batch][Hkv][2][R][D] or null
  const int32_t* page_table;     // [B][max_pages]
  const int32_t* seq_lens;       // [B], before the append
  int* status;
  int max_pages, B, T, Hkv, R, num_pages;
  int warps_per_group;           // ceil(B * T / 16)
  FastDiv div_wpg, div_T;        // division by warps_per_group and by T
  int cap_tokens;                // max_pages * 16, at most INT_MAX: a sequence fits
                                 // the page table while l0 <= cap_tokens - T
  int lq_w, lq_a, lq_rows;       // LogQuant base window W (0: off), log2 W, reserve rows
                                 // per plane; `window` is then the reserve
  int kpc;                       // key-per-channel mode: R is then the ring's R + 16 rows
  int lens_after;                // 1: seq_lens already count the T appended tokens
  LayerGeom geom;
};

struct DecodeParams {
  const uint8_t* pool;
  const uint16_t* window;        // bf16 ring or null
  const void* q;                 // [B][Hq][D] bf16 or fp32
  const int32_t* page_table;
  const int32_t* seq_lens;       // [B], including the window
  float* o;                      // fp32 [B][Hq][D]
  float* partials;               // fp32 [B][Hkv][NS][kMaxGroup][D + 2] (ticket mode)
  unsigned int* counters;        // [B][Hkv] tickets (ticket mode)
  int* status;
  int q_fp32, max_pages, B, Hq, Hkv, G, R, num_pages, had_block;
  int S;                         // quantized-token splits per (sequence, KV head)
  int NS;                        // S + the window or LogQuant reserve CTAs (0 to 4)
  int pages_per_split;       // host plan (page-table width / S); the kernel uses the lengths
  int overlap;               // launched with programmatic stream serialization
  int cluster;                   // 1: the NS (<= 4) CTAs of a unit merge in CTA 0's
                                 // shared memory -- a cluster when NS > 1, a lone CTA
                                 // combining its own partial when NS = 1; 0: tickets
  int step;                      // 1: decode step -- the new token (k_new, v_new) is
                                 // appended by this launch (seq_lens include it)
  const uint16_t* k_new;         // step: bf16 [B][Hkv][D]
  const uint16_t* v_new;
  int stage_bytes;               // bytes of one pipeline stage buffer
  float scale_log2;              // softmax_scale * log2(e)
  int lq_w, lq_a, lq_rows;       // LogQuant (as in AppendParams); R is 0 then, and the
                                 // split after the S quantized ones is the reserve's
  int wait_log2;                 // the main loop gives up on a page copy after
                                 // ~2^wait_log2 cycles (31 unless debugging)
  int kpc;                       // key-per-channel mode: per-channel K scales in the
                                 // pages; R is the ring's R + 16 rows; never a step
  LayerGeom geom;
};

// Decode kernel shape (build-time tuning knobs): warps per CTA, pipeline
// stages per warp, pages consumed per softmax round (1 or 2), and the minimum
// resident CTAs per SM the register allocation is sized for.
#ifndef KVQ_DECODE_WARPS
#define KVQ_DECODE_WARPS 4
#endif
#ifndef KVQ_DECODE_STAGES
#define KVQ_DECODE_STAGES 4
#endif
#ifndef KVQ_DECODE_ROUND
#define KVQ_DECODE_ROUND 2
#endif
#ifndef KVQ_DECODE_MIN_BLOCKS
#define KVQ_DECODE_MIN_BLOCKS 4
#endif
constexpr int kDecodeWarps = KVQ_DECODE_WARPS;
constexpr int kDecodeStages = KVQ_DECODE_STAGES;
constexpr int kDecodeRoundPages = KVQ_DECODE_ROUND;
constexpr int kDecodeMinBlocks = KVQ_DECODE_MIN_BLOCKS;
static_assert(kDecodeWarps >= 4, "the query prologue uses one warp per query head");
static_assert(kDecodeRoundPages == 1 || kDecodeRoundPages == 2, "1 or 2 pages per round");
static_assert(kDecodeStages % kDecodeRoundPages == 0, "stages are consumed a round at a time");
constexpr int kAppendWarps = 8;
// append: row buffers per warp (the chunk being quantized and the next one in
// flight; a third buffer measured slower) and resident CTAs per SM (the
// register allocation is sized for it)
constexpr int kAppendBufs = 2;
constexpr int kAppendCtas = 2;

// Launchers (defined in the .cu files).  Return cudaSuccess or the launch error.
cudaError_t launch_append(const AppendParams& p, int head_dim, int had_block, cudaStream_t s);
// LogQuant mode, before the append: the reserve's older members that the
// append's halvings thin move from the ring to their level buffers.
cudaError_t launch_lq_carry(const AppendParams& p, int head_dim, cudaStream_t s);
// Key-per-channel mode: quantizes the pages the append completes (keys per
// channel, values token-wise), then writes the positions that stay in bf16
// into the ring (two launches, in this order).
cudaError_t launch_kpc_append(const AppendParams& p, int head_dim, int had_block, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int head_dim, cudaStream_t s);
size_t decode_smem_bytes(const DecodeParams& p, int head_dim);
// resident CTAs per SM of the decode kernel (mode: 0 token-wise, 1 LogQuant,
// 2 key-per-channel), -1 on error
int decode_blocks_per_sm(int head_dim, size_t smem, int mode);
int decode_max_splits();
int decode_max_cluster();                               // largest cluster the merge uses

// Records `message` for kvq_last_error() on this thread and returns `status`.
kvq_status set_last_error(kvq_status status, const char* message);

}  // namespace kvq
