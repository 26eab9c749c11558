// Split-K decode attention over the paged quantized cache (sm_103a).
//
// Method: "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization for Real-World LLM
// Serving", section 3 (attention reads the compact cache; the rotation is undone
// on the fly -- here the query is rotated once, q . k = (H q) . (H k) / n, and
// the value accumulator is un-rotated once at the end, x = H u / n);
// "LogQuant ...", Methodology section 4 (A V = A_P V_P: partial results over any
// subsets of the tokens combine exactly, so splits, pages and the bf16 window
// are merged in any order) and section 2 (full-precision recent window).
//
// Grid (NS, Hkv, B): split s < S covers a contiguous range of quantized pages of
// sequence b for KV head h and its G <= 4 query heads; split S (when R > 0)
// covers the bf16 window, splits S .. NS - 1 the LogQuant reserve.  Each CTA merges its warps into one online-softmax
// partial (m, l, rotated acc[d] per query head).  Merge of the NS partials of a
// (b, h):
//   - cluster mode (NS <= 4): the NS CTAs form a thread-block cluster; each
//     CTA stores its partial straight into CTA 0's shared memory (distributed
//     shared memory), arrives on the cluster barrier and exits; CTA 0 waits on
//     the barrier, merges, un-rotates and writes o -- no global partials,
//     fences or atomics;
//   - ticket mode: partials go to global memory and the last CTA of (b, h) to
//     finish (an atomic ticket, no waiting) merges them.
//
// Quantized split, per warp: pages w, w + 4, ... of the split stream through a
// ring of shared-memory stages, each filled by one cp.async.bulk of a whole
// (page, head) segment (TMA engine, completion on an mbarrier).  A page is 16
// tokens = the M dimension of one m16n8k16 tensor-core MMA:
//   scores:  S[16 tok x 8] = C_K[16 tok x d] * Qhl[d x 8]
//   output:  O[d x 8]     += C_V^T[d x 16 tok] * Phl[16 tok x 8]
// where the 8 columns are the 4 query heads of the GQA group, each split into
// an fp16 "hi" part and an fp16 "lo" remainder (x = hi + lo to ~22 bits), so
// the group fills the n8 tile exactly and the fp32 accumulators keep fp32
// accuracy.  Codes enter the MMA as exact fp16 integers; the scale and zero are
// folded outside the MMA: score = s (q'' . c) + z sum(q''),
// sum_t p_t deq(v_t) = sum_t (p_t s_t) c_t + sum_t p_t z_t.
//
// The online softmax raises its running maximum only when a score passes it by
// more than a slack of 8 (log2 units) -- any maximum gives the same o = acc /
// l -- and redoes a round with the exact maximum when p s would leave fp16.
//
// Decode step (p.step): the warp owning the page of the new token quantizes it
// (the append's rule, bit for bit), writes it to the cache and patches its
// staged copy of the page, which it processes in its last round.
//
// Launch overlap (p.overlap, programmatic dependent launch): every CTA lets the
// next kernel launch at once; before griddepcontrol.wait a CTA reads only the
// page table, the lengths and the pool and starts its first copies; q, the new
// token and the window are read, and everything is written, after it.
#include <math_constants.h>

#include "kvq_logquant.h"
#include "kvq_quant.cuh"

namespace kvq {

namespace {

constexpr int kThreads = kDecodeWarps * 32;
// kernel instantiations: token-wise keys and values, LogQuant, key-per-channel
constexpr int kModeTokenWise = 0;
constexpr int kModeLogQuant = 1;
constexpr int kModeKeyChannel = 2;
constexpr int kMaxSplits = 256;
constexpr int kMaxCluster = 4;    // largest cluster the merge uses (CTA 0 holds its partials)
constexpr float kMaxSlack = 8.f;  // p <= 2^kMaxSlack under the lazy running maximum
constexpr float kMaxPS = 16384.f; // largest p s taken into an fp16 (hi, lo) pair

struct Smem {
  float* qtab;        // [kMaxGroup][D]   rotated query fragments (or raw query for the window)
  float* qsum;        // [kMaxGroup]
  int* flag;          // last-arriver flag of the ticket
  int* bad;           // a page id of this split was out of range
  int* wait_log2;     // the page-copy wait limit (a copy of p.wait_log2)
  float* qscl;        // [kMaxGroup] power-of-two scale of the query fragments
  uint64_t* bars;     // [warps][stages]
  float* merge;       // [warps][kMaxGroup][D + 2] warp partials
  float* cpart;       // [kMaxGroup * (D + 2)] this CTA's partial (layout as a global one)
  uint8_t* area;      // stage buffers / window scores
};

template <int D>
__host__ __device__ constexpr int merge_floats() { return kDecodeWarps * kMaxGroup * (D + 2); }

// CTAs whose partials CTA 0 gathers in shared memory: those of a cluster merge
// over more than one split (a single split combines its own partial).
__host__ __device__ constexpr int rbuf_ctas(int cluster, int ns) {
  return cluster && ns > 1 ? ns : 0;
}

// Bytes before the stage area: query fragments, a few words, the page-copy
// barriers, this CTA's partial, the cluster receive buffer of rbuf_ctas
// partials, and 128 bytes of slack for aligning the area.  The warps' merge
// region has no room of its own: it shares the stage area, and its first write
// comes after the barrier at which every warp is done with its stages (or with
// the window's rows), so that four CTAs of 8-bit keys with 4-bit values still
// fit an SM.
__host__ __device__ constexpr int header_bytes(int d, int rbuf_n) {
  return ((d * kMaxGroup * 4 + 64 + kDecodeWarps * kDecodeStages * 8 +
           (1 + rbuf_n) * kMaxGroup * (d + 2) * 4) +
          127) / 128 * 128 + 128;
}

template <int D>
__device__ __forceinline__ Smem carve(uint8_t* base, int rbuf_n) {
  Smem s;
  s.qtab = reinterpret_cast<float*>(base);
  uint8_t* misc = base + kMaxGroup * D * 4;
  s.qsum = reinterpret_cast<float*>(misc);
  s.flag = reinterpret_cast<int*>(misc + 16);
  s.bad = reinterpret_cast<int*>(misc + 20);
  s.wait_log2 = reinterpret_cast<int*>(misc + 24);
  s.qscl = reinterpret_cast<float*>(misc + 32);
  s.bars = reinterpret_cast<uint64_t*>(misc + 64);
  s.cpart = reinterpret_cast<float*>(misc + 64 + kDecodeWarps * kDecodeStages * 8);
  // then rbuf [rbuf_n][kMaxGroup * (D + 2)] (cluster mode, CTA 0: every CTA's
  // partial, pushed there through distributed shared memory; see rbuf())
  uint8_t* a = reinterpret_cast<uint8_t*>(s.cpart + (1 + rbuf_n) * kMaxGroup * (D + 2));
  s.area = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(a) + 127) & ~uintptr_t(127));
  s.merge = reinterpret_cast<float*>(s.area);
  return s;
}

// Cluster receive buffer (right after cpart).
template <int D>
__device__ __forceinline__ float* rbuf(const Smem& sm) { return sm.cpart + kMaxGroup * (D + 2); }

// A partial: acc [kMaxGroup][D] (fp32), then m [kMaxGroup] (log2 units) and
// l [kMaxGroup]; kMaxGroup * (D + 2) floats, rows 16-byte aligned.
template <int D>
__device__ __forceinline__ float* part_acc(float* part, int i) { return part + i * D; }
template <int D>
__device__ __forceinline__ const float* part_acc(const float* part, int i) { return part + i * D; }
template <int D>
__device__ __forceinline__ float* part_m(float* part) { return part + kMaxGroup * D; }
template <int D>
__device__ __forceinline__ const float* part_m(const float* part) { return part + kMaxGroup * D; }
template <int D>
__device__ __forceinline__ float* part_l(float* part) { return part + kMaxGroup * D + kMaxGroup; }
template <int D>
__device__ __forceinline__ const float* part_l(const float* part) {
  return part + kMaxGroup * D + kMaxGroup;
}

// Loads of NBYTES per lane from the shared-memory window (ld.shared, 32-bit
// address).  volatile keeps them after the mbarrier wait that guards the data.
template <int NBYTES>
__device__ __forceinline__ void lds_u32(uint32_t a, uint32_t* w) {
  if constexpr (NBYTES == 32) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(a));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "r"(a + 16));
  } else if constexpr (NBYTES == 16) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(a));
  } else if constexpr (NBYTES == 8) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(a));
  } else if constexpr (NBYTES == 4) {
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[0]) : "r"(a));
  } else {
    static_assert(NBYTES == 2, "unsupported row slice");
    uint16_t x;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(x) : "r"(a));
    w[0] = x;
  }
}

__device__ __forceinline__ float2 lds_half2(uint32_t a) {
  uint32_t x;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(a));
  return __half22float2(*reinterpret_cast<const __half2*>(&x));
}

// ------------------------------------------------- K codes -> fp16 pairs ----
// Exact fp16 integers: a code's bits OR-ed into the mantissa of 1024.0 give
// 1024 + c * 2^k (k its bit position), brought back to c by one packed fp16
// subtract or multiply-add.  (Feeding 1024 + c * 2^k to the MMA and taking the
// offset off afterwards would save that instruction, but the offset inflates
// the fp32 partial sums of the MMA by up to ~100x, which costs too much score
// precision on keys with large outlier channels.)
// K pair i: dims kpair_dims() of one token row (w: the lane's slice of it).
// Each pair is formed right before the MMA that takes it.
template <int BITS>
__device__ __forceinline__ uint32_t kpair(const uint32_t* w, int i) {
  if constexpr (BITS == 4) {
    const uint32_t x = (i & 2) ? (w[i >> 2] >> 8) : w[i >> 2];
    return (i & 1) ? h2_unscale<4>(lop_or_magic(x, 0x00f000f0u))
                   : h2_sub1024(lop_or_magic(x, 0x000f000fu));
  } else if constexpr (BITS == 2) {
    const int k = i & 7;
    const uint32_t x = (k & 4) ? (w[i >> 3] >> 8) : w[i >> 3];
    switch (k & 3) {
      case 0: return h2_sub1024(lop_or_magic(x, 0x00030003u));
      case 1: return h2_unscale<2>(lop_or_magic(x, 0x000c000cu));
      case 2: return h2_unscale<4>(lop_or_magic(x, 0x00300030u));
      default: return h2_unscale<6>(lop_or_magic(x, 0x00c000c0u));
    }
  } else {
    return h2_sub1024(__byte_perm(w[i >> 1], 0x64646464u, (i & 1) ? 0x4342 : 0x4140));
  }
}

// Key-per-channel mode: the stored field is c + 2^(BITS-1) (offset binary);
// the same LOP3 and one HSUB / HFMA whose constant also takes off 2^(BITS-1)
// give the signed code c exactly.
__device__ __forceinline__ uint32_t h2_sub(uint32_t x, float c) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), __half2(__half(c), __half(c)));
  return *reinterpret_cast<uint32_t*>(&r);
}
template <int K>
__device__ __forceinline__ uint32_t h2_unscale_off(uint32_t x, float off) {
  constexpr float inv = 1.0f / float(1 << K);
  const float c = -1024.0f / float(1 << K) - off;
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), __half2(__half(inv), __half(inv)),
                      __half2(__half(c), __half(c)));
  return *reinterpret_cast<uint32_t*>(&r);
}
template <int BITS>
__device__ __forceinline__ uint32_t kpair_signed(const uint32_t* w, int i) {
  constexpr float off = float(1 << (BITS - 1));
  if constexpr (BITS == 4) {
    const uint32_t x = (i & 2) ? (w[i >> 2] >> 8) : w[i >> 2];
    return (i & 1) ? h2_unscale_off<4>(lop_or_magic(x, 0x00f000f0u), off)
                   : h2_sub(lop_or_magic(x, 0x000f000fu), 1024.f + off);
  } else if constexpr (BITS == 2) {
    const int k = i & 7;
    const uint32_t x = (k & 4) ? (w[i >> 3] >> 8) : w[i >> 3];
    switch (k & 3) {
      case 0: return h2_sub(lop_or_magic(x, 0x00030003u), 1024.f + off);
      case 1: return h2_unscale_off<2>(lop_or_magic(x, 0x000c000cu), off);
      case 2: return h2_unscale_off<4>(lop_or_magic(x, 0x00300030u), off);
      default: return h2_unscale_off<6>(lop_or_magic(x, 0x00c000c0u), off);
    }
  } else {
    return h2_sub(__byte_perm(w[i >> 1], 0x64646464u, (i & 1) ? 0x4342 : 0x4140), 1024.f + off);
  }
}

// (low dim, high dim) of K pair i for k-slot group c; dims of the thread's
// quarter [c * D / 4, (c + 1) * D / 4) of the row.
template <int D, int BITS>
__device__ __forceinline__ void kpair_dims(int c, int i, int& lo, int& hi) {
  const int base = c * (D / 4);
  if constexpr (BITS == 4) {
    lo = base + 8 * (i >> 2) + (i & 3);
    hi = lo + 4;
  } else if constexpr (BITS == 2) {
    lo = base + 16 * (i >> 3) + (i & 7);
    hi = lo + 8;
  } else {
    lo = base + 4 * (i >> 1) + 2 * (i & 1);
    hi = lo + 1;
  }
}

// ------------------------------------- V codes of two tokens -> fp16 pairs --
// V pair i: dim i of the lane's slice for two tokens (w1 in the low half, w2
// high): the rows' bytes interleaved, then the same masks as for K.
template <int BITS>
__device__ __forceinline__ uint32_t vpair(const uint32_t* w1, const uint32_t* w2, int i) {
  if constexpr (BITS == 4) {
    const int k = i & 7;
    const uint32_t ab = __byte_perm(w1[i >> 3], w2[i >> 3], (k & 4) ? 0x7632 : 0x5410);
    const uint32_t x = (k & 2) ? (ab >> 8) : ab;
    return (k & 1) ? h2_unscale<4>(lop_or_magic(x, 0x00f000f0u))
                   : h2_sub1024(lop_or_magic(x, 0x000f000fu));
  } else if constexpr (BITS == 2) {
    // a word holds 16 dims; the 2-byte slice (head_dim 64) holds 8
    const int k = i & 15;
    const uint32_t ab = __byte_perm(w1[i >> 4], w2[i >> 4], (k & 8) ? 0x7632 : 0x5410);
    const uint32_t x = (k & 4) ? (ab >> 8) : ab;
    switch (k & 3) {
      case 0: return h2_sub1024(lop_or_magic(x, 0x00030003u));
      case 1: return h2_unscale<2>(lop_or_magic(x, 0x000c000cu));
      case 2: return h2_unscale<4>(lop_or_magic(x, 0x00300030u));
      default: return h2_unscale<6>(lop_or_magic(x, 0x00c000c0u));
    }
  } else {
    const uint32_t sel = 0x4400u + 0x1111u * static_cast<uint32_t>(i & 3);
    return h2_sub1024(lop_or_magic(__byte_perm(w1[i >> 2], w2[i >> 2], sel), 0x00ff00ffu));
  }
}

__device__ __forceinline__ float warp_max_group(float x) {  // over lanes with equal lane % 4
  x = fmaxf(x, __shfl_xor_sync(kFullMask, x, 4));
  x = fmaxf(x, __shfl_xor_sync(kFullMask, x, 8));
  return fmaxf(x, __shfl_xor_sync(kFullMask, x, 16));
}
__device__ __forceinline__ float warp_sum_group(float x) {
  x += __shfl_xor_sync(kFullMask, x, 4);
  x += __shfl_xor_sync(kFullMask, x, 8);
  return x + __shfl_xor_sync(kFullMask, x, 16);
}

__device__ __forceinline__ float hi_part(float x) { return __half2float(__float2half_rn(x)); }

// ------------------------------------------------------- query prologue --
// Per-warp register layout of one D-vector: lane l holds dims [E l, E l + E),
// E = D / 32.  Warp i < G loads query head h * G + i of sequence b (zeros for
// i >= G), exactly (bf16 or fp32 to fp32).
__device__ __forceinline__ uint32_t ldg_nc_u32(const void* ptr) {
  uint32_t x;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(x) : "l"(ptr));
  return x;
}
__device__ __forceinline__ uint32_t ldg_nc_u16(const void* ptr) {
  uint16_t x;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(x) : "l"(ptr));
  return x;
}

template <int D>
__device__ __forceinline__ void load_query(const DecodeParams& p, int b, int h, float (&v)[D / 32]) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = 0.f;
  if (warp < p.G) {
    const size_t off = (static_cast<size_t>(b) * p.Hq + h * p.G + warp) * D + E * lane;
    if (p.q_fp32) {
#pragma unroll
      for (int e = 0; e < E; ++e)
        v[e] = __uint_as_float(ldg_nc_u32(reinterpret_cast<const float*>(p.q) + off + e));
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e)
        v[e] = __uint_as_float(ldg_nc_u16(reinterpret_cast<const uint16_t*>(p.q) + off + e) << 16);
    }
  }
}

// First chunk of this warp's page ids (pages pg0 + warp + 4 k, k < 32, lane
// k), bounded by the page-table row only, so that it can be issued before the
// sequence length is known; 0 past the row.
__device__ __forceinline__ int load_page_chunk0(const DecodeParams& p, int b, int pg0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pg = pg0 + warp + kDecodeWarps * lane;
  if (pg >= p.max_pages) return 0;
  return static_cast<int>(ldg_nc_u32(p.page_table + static_cast<size_t>(b) * p.max_pages + pg));
}

// Unnormalised block-diagonal Sylvester transform (blocks of nb) of a D-vector
// held in the per-warp layout: stage hs adds and subtracts the elements
// (i, i + hs) of every block, first inside a lane, then across lanes.
template <int E>
__device__ __forceinline__ void warp_fwht(float (&v)[E], int nb) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int hs = 1; hs < E; hs <<= 1) {
    if (hs >= nb) break;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (!(e & hs)) {
        const float a = v[e], c = v[e + hs];
        v[e] = a + c;
        v[e + hs] = a - c;
      }
    }
  }
  for (int m = 1; m * E < nb; m <<= 1) {  // partner lane = lane ^ m
    const bool upper = lane & m;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(kFullMask, v[e], m);
      v[e] = upper ? o - v[e] : v[e] + o;
    }
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFullMask, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFullMask, x, o));
  return x;
}

// 2^x with the hardware approximation (relative error ~2^-22); 2^-inf = 0
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp16 (hi, lo) split of x: hi = fp16(x) in the low half, lo = fp16(x - hi) high.
__device__ __forceinline__ uint32_t hilo_pair(float x) {
  const float hi = hi_part(x);
  const __half2 r = __floats2half2_rn(x, x - hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Quantized splits: q'' = (H q / n) * softmax_scale * log2(e) for each query
// head of the group (warp i: head i).  A power-of-two scale e_i puts
// max_d |q''| in [2^13, 2^14), so that both fp16 parts of x = e_i q''_d
// (hi = fp16(x), lo = fp16(x - hi)) stay normal and together carry ~22 bits
// of x.  Writes qtab[i][d] = the packed pair (hi, lo) (as raw bits),
// qsum[i] = e_i sum_d q''_d and qscl[i] = 1 / e_i.
// RAW (key-per-channel mode): qtab[i][d] = e_i q''_d as fp32 instead of the
// packed pair; the B fragments are formed per page with its channel scales.
template <int D, bool RAW = false>
__device__ void query_quant_prologue(const DecodeParams& p, const Smem& sm, float (&v)[D / 32]) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kMaxGroup) {
    __syncthreads();
    return;
  }
  warp_fwht<E>(v, p.had_block);
  const float qscale = p.scale_log2 / static_cast<float>(p.had_block);
  float s = 0.f, amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    v[e] *= qscale;
    s += v[e];
    amax = fmaxf(amax, fabsf(v[e]));
  }
  s = warp_sum(s);
  amax = warp_max(amax);
  int ex = 13;
  if (amax > 0.f && isfinite(amax)) {
    const int e2 = ((__float_as_int(amax) >> 23) & 0xff) - 127;   // amax in [2^e2, 2^(e2+1))
    ex = max(-100, min(100, 13 - e2));
  }
  const float scl = ldexpf(1.f, ex);
  uint32_t* qt = reinterpret_cast<uint32_t*>(sm.qtab) + warp * D + E * lane;
#pragma unroll
  for (int e = 0; e < E; ++e) qt[e] = RAW ? __float_as_uint(v[e] * scl) : hilo_pair(v[e] * scl);
  if (lane == 0) {
    sm.qsum[warp] = s * scl;
    sm.qscl[warp] = ldexpf(1.f, -ex);
  }
  __syncthreads();
}

// Window split: qtab[i][d] = q_d * softmax_scale * log2(e), not rotated.
template <int D>
__device__ void query_window_prologue(const DecodeParams& p, const Smem& sm, const float (&v)[D / 32]) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < kMaxGroup) {
#pragma unroll
    for (int e = 0; e < E; ++e) sm.qtab[warp * D + E * lane + e] = v[e] * p.scale_log2;
  }
  __syncthreads();
}

// ------------------------------------------------------------ quantized split
// movmatrix: 8x8 transpose of 16-bit elements across the warp.  In: lane
// (g, c) holds row g, columns (2c, 2c+1); out: row g of the transpose.
__device__ __forceinline__ uint32_t movm_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Programmatic dependent launch.  launch_dependents lets the next kernel on
// the stream start its CTAs early; wait returns once the kernel launched before
// this one has completed and its writes are visible (at once when this grid was
// launched without programmatic stream serialization).
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// CTA merge, warp i: the partials of query head i of the kDecodeWarps warps
// (merge region) -> the CTA's partial of head i in `out`; `drop` empties it.
template <int D>
__device__ __forceinline__ void merge_warps(const Smem& sm, int i, bool drop, float* out) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const float* macc = sm.merge;
  const float* mml = macc + kDecodeWarps * kMaxGroup * D;
  float mw[kDecodeWarps], mm = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < kDecodeWarps; ++w) {
    mw[w] = drop ? -CUDART_INF_F : mml[w * kMaxGroup + i];
    mm = fmaxf(mm, mw[w]);
  }
  float acc[E], ll = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
  for (int w = 0; w < kDecodeWarps; ++w) {
    const float f = mw[w] == -CUDART_INF_F ? 0.f : ex2(mw[w] - mm);
    if (f != 0.f) {
      ll = __fmaf_rn(f, mml[kDecodeWarps * kMaxGroup + w * kMaxGroup + i], ll);
      const float* row = macc + (w * kMaxGroup + i) * D + E * lane;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(f, row[e], acc[e]);
    }
  }
  float* dst = part_acc<D>(out, i) + E * lane;
#pragma unroll
  for (int e = 0; e < E; ++e) dst[e] = acc[e];
  if (lane == 0) {
    part_m<D>(out)[i] = mm;
    part_l<D>(out)[i] = ll;
  }
}

// ------------------------------------------------------------ decode step --
// This lane's part of the decode step's new token, loaded at kernel start:
// lanes 0-15 hold K elements [F l, F l + F), lanes 16-31 the same of V
// (F = D / 16), as packed bf16 pairs.
template <int D>
__device__ __forceinline__ void load_new_token(const DecodeParams& p, int b, int h,
                                               uint32_t (&w)[D / 32]) {
  constexpr int F = D / 16;
  const int lane = threadIdx.x & 31;
  const uint16_t* src = (lane < 16 ? p.k_new : p.v_new) +
                        (static_cast<size_t>(b) * p.Hkv + h) * D + F * (lane & 15);
#pragma unroll
  for (int i = 0; i < F / 2; ++i) w[i] = ldg_nc_u32(src + 2 * i);
}

// Stores n = F * bits / 8 bytes (1, 2, 4 or 8; naturally aligned) of codes.
__device__ __forceinline__ void store_codes(uint8_t* dst, const uint32_t (&c)[2], int n) {
  if (n == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(c[0], c[1]);
  else if (n == 4) *reinterpret_cast<uint32_t*>(dst) = c[0];
  else if (n == 2) *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(c[0]);
  else *dst = static_cast<uint8_t>(c[0]);
}

// Decode step, the warp that owns page pos / 16 (pos = the last quantized
// position): quantizes the K (lanes 0-15) and V (lanes 16-31) vectors of
// position pos -- the new token itself without a window; with one, the token
// that leaves the ring now, whose slot then takes the new token -- and writes
// them to the cache page (for later calls) and to `pbuf` in shared memory
// (K codes [KB], V codes [VB], K (s, z), V (s, z)), from which this launch's
// staged copy of the page gets patched.  Same rule and same bits as kvq_append.
// pid: the page table's entry for that page (read by the caller before the
// launch-overlap wait; an id outside [0, num_pages) is reported and not written).
template <int D>
__device__ void step_append(const DecodeParams& p, int b, int h, int pos, int bk, int bv,
                            const uint32_t (&tok)[D / 32], uint8_t* pbuf, int pid) {
  constexpr int F = D / 16;
  const int lane = threadIdx.x & 31, half = lane >> 4, l = lane & 15;
  const int bits = half ? bv : bk;
  const int KB = D * bk / 8, VB = D * bv / 8;
  const int rowb = half ? VB : KB;              // code bytes of this vector's row
  const int nb = F * bits / 8;                  // code bytes of this lane
  uint16_t* ring = nullptr;                     // this lane's elements of the ring slot
  if (p.R > 0)
    ring = const_cast<uint16_t*>(p.window) + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + half) *
                                                  p.R * D +
           static_cast<size_t>(pos % p.R) * D + F * l;
  float v[F];
  if (ring) {                                   // the token leaving the ring
#pragma unroll
    for (int i = 0; i < F / 2; ++i) {
      const uint32_t x = *reinterpret_cast<const uint32_t*>(ring + 2 * i);
      v[2 * i] = bf16lo(x);
      v[2 * i + 1] = bf16hi(x);
    }
  } else {
#pragma unroll
    for (int i = 0; i < F / 2; ++i) {
      v[2 * i] = bf16lo(tok[i]);
      v[2 * i + 1] = bf16hi(tok[i]);
    }
  }
  uint32_t codes[2];
  __half sh, zh;
  rotate_quantize_halfwarp<D>(v, p.had_block, bits, codes, sh, zh);
  uint8_t* seg = nullptr;
  if (pid >= 0 && pid < p.num_pages) {
    seg = const_cast<uint8_t*>(p.pool) + static_cast<size_t>(pid) * p.geom.page_bytes +
          p.geom.head_off[h];
  } else if (lane == 0) {
    flag_status(p.status, KVQ_DEV_BAD_PAGE);
  }
  const int slot = pos % kPage;
  store_codes(pbuf + (half ? KB : 0) + nb * l, codes, nb);
  if (seg) store_codes(seg + (half ? kPage * KB : 0) + slot * rowb + nb * l, codes, nb);
  if (l == 0) {
    if (!(isfinite(__half2float(sh)) && isfinite(__half2float(zh))))
      flag_status(p.status, KVQ_DEV_NONFINITE);
    const uint32_t sz = pack_half2(sh, zh);
    *reinterpret_cast<uint32_t*>(pbuf + KB + VB + 4 * half) = sz;
    if (seg) *reinterpret_cast<uint32_t*>(seg + kPage * (KB + VB) + 4 * kPage * half + slot * 4) = sz;
  }
  if (ring) {                                   // the new token takes the slot
#pragma unroll
    for (int i = 0; i < F / 2; ++i) *reinterpret_cast<uint32_t*>(ring + 2 * i) = tok[i];
  }
  __syncwarp();
}

// Copies the patch (step_append's pbuf) into slot `slot` of the staged page
// at shared-window address st, once its copy has landed.
template <int D, int BK, int BV>
__device__ __forceinline__ void patch_stage(uint32_t st, const uint8_t* pbuf, int slot) {
  constexpr int KB = D * BK / 8, VB = D * BV / 8;
  const int lane = threadIdx.x & 31;
  const uint32_t src = smem_u32(pbuf);
  for (int w = lane; w < (KB + VB) / 4 + 2; w += 32) {
    uint32_t x;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(src + 4 * w));
    uint32_t dst;
    if (w < KB / 4) dst = st + slot * KB + 4 * w;
    else if (w < (KB + VB) / 4) dst = st + kPage * KB + slot * VB + 4 * w - KB;
    else if (w == (KB + VB) / 4) dst = st + kPage * (KB + VB) + slot * 4;
    else dst = st + kPage * (KB + VB) + 4 * kPage + slot * 4;
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(dst), "r"(x) : "memory");
  }
  // these generic writes come before any later bulk copy into the stage
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// One split of one (sequence, KV head): pages [split * pps, (split + 1) * pps)
// of the quantized part; warp w takes pages w, w + 4, ... two at a time.
// LQ: LogQuant mode -- the members of B (full precision, attended by the
// reserve split) are left out here, on the rounds whose pages can hold one.
template <int D, int BK, int BV, int MODE>
__device__ void quant_split(const DecodeParams& p, const Smem& sm, int b, int h, int split,
                            int lq, int len, float (&qv)[D / 32], int chunk0,
                            uint32_t (&tok)[D / 32]) {
  constexpr bool LQ = MODE == kModeLogQuant;
  constexpr bool KPC = MODE == kModeKeyChannel;
  constexpr int KB = D * BK / 8;                 // K code bytes per token
  constexpr int VB = D * BV / 8;
  // one (page, head) segment: codes, then K (s, z) per token or K scales per
  // channel, then V (s, z) per token
  constexpr int CHUNK = KPC ? kPage * (KB + VB) + 2 * D + 4 * kPage : kPage * (KB + VB + 8);
  constexpr int NJ = D / 16;                     // MMAs along d
  constexpr int KSLICE = KB / 4;                 // bytes of a token row per k-slot group
  constexpr int VSLICE = VB / 8;                 // bytes of a token row per dim group
  constexpr int KWORDS = KSLICE >= 4 ? KSLICE / 4 : 1;
  constexpr int VWORDS = VSLICE >= 4 ? VSLICE / 4 : 1;
  // pairs of the lane's V slice (>= 2 * NJ; only head_dim 64 with 2-bit values
  // has more, from the zero upper half of a 2-byte slice)
  static_assert((BV == 2 ? 16 : BV == 4 ? 8 : 4) * VWORDS >= 2 * NJ, "value slice too small");
  constexpr int NST = kDecodeStages;
  static_assert(NST % 2 == 0, "stages are consumed in pairs");
  constexpr uint32_t KSZ = kPage * (KB + VB);    // offset of the K (s, z) pairs or scales
  constexpr uint32_t VSZ = KSZ + (KPC ? 2 * D : 4 * kPage);  // offset of the V (s, z) pairs

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int num_pages = p.num_pages;
  const uint32_t stage_bytes = static_cast<uint32_t>(p.stage_bytes);

  // ---- this warp's pages: first + 4 k, k < nk; their ids in registers,
  //      32 per chunk (lane i holds page k = 32 * chunk + i).  Ids outside
  //      [0, num_pages) are reported, replaced by page 0 so that every copy
  //      stays in bounds, and the whole split is dropped at the end.
  // S splits of this sequence's pages: the host plan's split size (from the
  // page-table width) while it still gives every split pages, else the split
  // size of this length (and the page ids loaded for the plan's are reloaded)
  const int npages = (lq + kPage - 1) / kPage;
  const int pps = npages > p.pages_per_split * (p.S - 1) ? p.pages_per_split
                                                          : max(1, (npages + p.S - 1) / p.S);
  const int pg0 = split * pps;
  const int pg1 = min(npages, pg0 + pps);
  if (pps != p.pages_per_split) chunk0 = load_page_chunk0(p, b, pg0);
  const int first = pg0 + warp;
  const int nk = pg1 > first ? (pg1 - first + kDecodeWarps - 1) / kDecodeWarps : 0;
  const int32_t* ptab = p.page_table + static_cast<size_t>(b) * p.max_pages + first;
  auto check_chunk = [&](int ch, int pid) -> int {
    const int kk = 32 * ch + lane;
    if (kk >= nk) pid = 0;
    const bool bad = pid < 0 || pid >= num_pages;
    if (__any_sync(kFullMask, bad)) {
      if (bad) {
        flag_status(p.status, KVQ_DEV_BAD_PAGE);
        *reinterpret_cast<volatile int*>(sm.bad) = 1;
      }
      if (bad) pid = 0;
    }
    return pid;
  };
  auto load_chunk = [&](int ch) -> int {
    const int kk = 32 * ch + lane;
    return check_chunk(ch, kk < nk ? __ldg(ptab + kDecodeWarps * kk) : 0);
  };
  int chunk = 0;
  int pid_cur = check_chunk(0, chunk0);
  int pid_nxt = nk > 32 ? load_chunk(1) : 0;
  auto pid_of = [&](int kk) -> int {  // warp-uniform kk in [32 chunk, 32 chunk + 64)
    const int v = (kk >> 5) == chunk ? pid_cur : pid_nxt;
    return __shfl_sync(kFullMask, v, kk & 31);
  };
  uint8_t* stages = sm.area + static_cast<size_t>(warp) * NST * stage_bytes;
  const uint32_t st0 = smem_u32(stages);        // shared-window address of stage 0
  uint64_t* bars = sm.bars + warp * NST;
  const uint8_t* head_base = p.pool + p.geom.head_off[h];
  // a page holds at most 64 heads' segments (< 1 MB): its byte offset is one
  // 32 x 32 -> 64-bit multiply-add per copy
  const uint32_t page_bytes = static_cast<uint32_t>(p.geom.page_bytes);
  // lane 0 issues the copy of page `pid` (already validated) into `slot` when
  // `go` (predicated, no branch)
  const uint32_t bars0 = smem_u32(bars);
  auto issue = [&](bool go, int slot, int pid) {
    bulk_g2s_if(go && lane == 0, st0 + slot * stage_bytes,
                head_base + static_cast<uint32_t>(pid) * static_cast<size_t>(page_bytes), CHUNK,
                bars0 + 8u * slot);
  };
  // start streaming before the query prologue (with a shortened copy wait, a
  // debugging aid, only right before the loop: the first waits then come
  // sooner than any copy can land)
  if (p.wait_log2 >= kWaitLimitLog2)
    for (int kk = 0; kk < nk && kk < NST; ++kk) issue(true, kk, pid_of(kk));

  // decode step: the warp owning the page of the last quantized position
  // quantizes the token there (after the wait) while its first copies are in
  // flight; that page's id is read now (the page table is an input)
  int kpatch = -1, step_pid = -1;
  if (!KPC && p.step && lq > 0) {   // (the key-per-channel mode appends before the launch)
    const int pl = npages - 1;
    if (pl >= pg0 && pl < pg1 && (pl - pg0) % kDecodeWarps == warp) {
      kpatch = (pl - pg0) / kDecodeWarps;
      step_pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pl);
    }
  }

  // with programmatic dependent launch, everything above may overlap the
  // previous kernel; q and the new token are its results
  grid_wait();
  if (p.overlap) {
    load_query<D>(p, b, h, qv);
    if (p.step) load_new_token<D>(p, b, h, tok);
  }

  uint8_t* pbuf = reinterpret_cast<uint8_t*>(sm.cpart);   // free until the warps merge
  if (kpatch >= 0) step_append<D>(p, b, h, lq - 1, BK, BV, tok, pbuf, step_pid);
  const int pslot = (lq - 1) % kPage;

  // key-per-channel codes of 2 bits are -1, 0 or 1, so c s is exact in fp16:
  // the page's scales go into the A operand and the query keeps its constant
  // B fragments (KPC2); wider codes form B per page from fp32 queries
  constexpr bool KPC2 = KPC && BK == 2;
  // 4-bit codes (|c| <= 7) take the page's scales split in two exact parts
  constexpr bool KPC4 = KPC && BK == 4;
  query_quant_prologue<D, KPC && !KPC2 && !KPC4>(p, sm, qv);

  // ---- B fragments of the K-side MMA: column n = g is query head g / 2, its
  //      hi part for even g and lo part for odd g (per page in the
  //      key-per-channel mode)
  uint32_t bq[NJ][2];
  if constexpr (!KPC || KPC2 || KPC4) {
    const uint32_t* qh = reinterpret_cast<const uint32_t*>(sm.qtab) + (g >> 1) * D;
    const int sh = (g & 1) ? 16 : 0;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        int d0, d1;
        kpair_dims<D, BK>(c, 2 * j + s2, d0, d1);
        bq[j][s2] = ((qh[d0] >> sh) & 0xffffu) | (((qh[d1] >> sh) & 0xffffu) << 16);
      }
    }
  }
  const float qs = sm.qsum[c];          // scaled sum of the query (head c)
  const float iscl = sm.qscl[c];        // scores are scaled by 1 / iscl

  // running softmax state of head c in scaled units: m_s = m / iscl
  float m_s = -CUDART_INF_F, mneg = CUDART_INF_F;  // mneg = -m (true units)
  float l = 0.f, zacc = 0.f;
  float oacc[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

  // per-lane offsets inside a stage
  const uint32_t koff = g * KB + c * KSLICE;                       // K row g, slice c
  const uint32_t voff = kPage * KB + g * VSLICE + 2 * c * VB;      // V row 2c, slice g

  // scaled scores of tokens (g, g + 8) of the page staged at `st`
  auto scores = [&](uint32_t st, float& sc0, float& sc1) {
    uint32_t w0[KWORDS], w1[KWORDS];
    lds_u32<KSLICE>(st + koff, w0);
    lds_u32<KSLICE>(st + koff + 8 * KB, w1);
    const float2 k0 = lds_half2(st + KSZ + 4 * g);
    const float2 k1 = lds_half2(st + KSZ + 4 * g + 32);
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const uint32_t x[4] = {kpair<BK>(w0, 2 * j), kpair<BK>(w1, 2 * j),
                             kpair<BK>(w0, 2 * j + 1), kpair<BK>(w1, 2 * j + 1)};
      mma_16816(a, x, bq[j][0], bq[j][1]);
    }
    sc0 = __fmaf_rn(k0.x, a[0] + a[1], k0.y * qs);
    sc1 = __fmaf_rn(k1.x, a[2] + a[3], k1.y * qs);
  };
  // key-per-channel mode: score = sum_d (e q''_d) s_d c_d with the page's
  // channel scales s_d.  Column g of the B fragments takes head g / 2's
  // x_d = (e q''_d)(s_d 2^-E), hi part (even g) or lo part (odd g), where 2^E
  // is the binade of the page's largest scale (x < 2^15 stays inside fp16);
  // the scaled score is (a0 + a1) 2^E.  Codes are signed, no zero term.
  constexpr int QD = D / 4;                      // dims of a k-slot group
  // 2-bit key-per-channel: A = c s_d (exact), B the constant query fragments;
  // the scaled score is a_hi + a_lo (no zero term)
  auto scores_kpc2 = [&](uint32_t st, float& sc0, float& sc1) {
    uint32_t w0[KWORDS], w1[KWORDS];
    lds_u32<KSLICE>(st + koff, w0);
    lds_u32<KSLICE>(st + koff + 8 * KB, w1);
    uint32_t sw[QD / 2];                         // scales of dims [c QD, (c + 1) QD)
#pragma unroll
    for (int i = 0; i < QD / 16; ++i) lds_u32<32>(st + KSZ + c * (QD * 2) + 32 * i, sw + 8 * i);
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      uint32_t sp[2];
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        int d0, d1;
        kpair_dims<D, BK>(0, 2 * j + s2, d0, d1);
        sp[s2] = __byte_perm(sw[d0 >> 1], sw[d1 >> 1],
                             ((d0 & 1) ? 0x0032u : 0x0010u) | ((d1 & 1) ? 0x7600u : 0x5400u));
      }
      auto scaled = [&](uint32_t code2, uint32_t s2v) -> uint32_t {
        const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&code2),
                                  *reinterpret_cast<const __half2*>(&s2v));
        return *reinterpret_cast<const uint32_t*>(&r);
      };
      const uint32_t x[4] = {scaled(kpair_signed<BK>(w0, 2 * j), sp[0]),
                             scaled(kpair_signed<BK>(w1, 2 * j), sp[0]),
                             scaled(kpair_signed<BK>(w0, 2 * j + 1), sp[1]),
                             scaled(kpair_signed<BK>(w1, 2 * j + 1), sp[1])};
      mma_16816(a, x, bq[j][0], bq[j][1]);
    }
    sc0 = a[0] + a[1];
    sc1 = a[2] + a[3];
  };
  // 4-bit key-per-channel: the page's scales, normalised by 2^-E (2^E the
  // binade of the largest, so every s' < 2), split as s' = s_hi + s_lo with
  // s_hi keeping 8 significant bits and s_lo the other 3: c s_hi and c s_lo
  // (|c| <= 7) are exact in fp16, and two MMAs against the constant query
  // fragments give sum_d c s'_d q_d; the scaled score is (a_hi + a_lo) 2^E
  auto scores_kpc4 = [&](uint32_t st, float& sc0, float& sc1) {
    uint32_t w0[KWORDS], w1[KWORDS];
    lds_u32<KSLICE>(st + koff, w0);
    lds_u32<KSLICE>(st + koff + 8 * KB, w1);
    uint32_t sw[QD / 2];                         // scales of dims [c QD, (c + 1) QD)
#pragma unroll
    for (int i = 0; i < QD / 16; ++i) lds_u32<32>(st + KSZ + c * (QD * 2) + 32 * i, sw + 8 * i);
    uint32_t mx = sw[0];                         // scales are >= 0: fp16 bits order them
#pragma unroll
    for (int i = 1; i < QD / 2; ++i) mx = __vmaxu2(mx, sw[i]);
    mx = max(mx & 0xffffu, mx >> 16);
    mx = max(mx, __shfl_xor_sync(kFullMask, mx, 1));
    mx = max(mx, __shfl_xor_sync(kFullMask, mx, 2));
    const int ex = max(static_cast<int>(mx >> 10), 1) - 15;    // subnormal: -14
    const float up = __int_as_float((127 + ex) << 23);
    const unsigned dh = -ex >= -14 ? static_cast<unsigned>(15 - ex) << 10 : 1u << (24 - ex);
    const uint32_t down2 = dh | (dh << 16);
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      uint32_t shi[2], slo[2];
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        int d0, d1;
        kpair_dims<D, BK>(0, 2 * j + s2, d0, d1);
        uint32_t sp = __byte_perm(sw[d0 >> 1], sw[d1 >> 1],
                                  ((d0 & 1) ? 0x0032u : 0x0010u) | ((d1 & 1) ? 0x7600u : 0x5400u));
        __half2 sn = __hmul2(*reinterpret_cast<const __half2*>(&sp),
                             *reinterpret_cast<const __half2*>(&down2));
        const uint32_t snb = *reinterpret_cast<const uint32_t*>(&sn);
        shi[s2] = snb & 0xfff8fff8u;             // the low 3 mantissa bits cleared
        const __half2 lo = __hsub2(sn, *reinterpret_cast<const __half2*>(&shi[s2]));
        slo[s2] = *reinterpret_cast<const uint32_t*>(&lo);
      }
      auto scaled = [&](uint32_t code2, uint32_t s2v) -> uint32_t {
        const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&code2),
                                  *reinterpret_cast<const __half2*>(&s2v));
        return *reinterpret_cast<const uint32_t*>(&r);
      };
      const uint32_t c00 = kpair_signed<BK>(w0, 2 * j), c10 = kpair_signed<BK>(w1, 2 * j);
      const uint32_t c01 = kpair_signed<BK>(w0, 2 * j + 1), c11 = kpair_signed<BK>(w1, 2 * j + 1);
      const uint32_t xh[4] = {scaled(c00, shi[0]), scaled(c10, shi[0]), scaled(c01, shi[1]),
                              scaled(c11, shi[1])};
      const uint32_t xl[4] = {scaled(c00, slo[0]), scaled(c10, slo[0]), scaled(c01, slo[1]),
                              scaled(c11, slo[1])};
      mma_16816(a, xh, bq[j][0], bq[j][1]);
      mma_16816(a, xl, bq[j][0], bq[j][1]);
    }
    sc0 = (a[0] + a[1]) * up;
    sc1 = (a[2] + a[3]) * up;
  };
  auto scores_kpc = [&](uint32_t st, float& sc0, float& sc1) {
    uint32_t w0[KWORDS], w1[KWORDS];
    lds_u32<KSLICE>(st + koff, w0);
    lds_u32<KSLICE>(st + koff + 8 * KB, w1);
    uint32_t sw[QD / 2];                         // scales of dims [c QD, (c + 1) QD)
#pragma unroll
    for (int i = 0; i < QD / 16; ++i) lds_u32<32>(st + KSZ + c * (QD * 2) + 32 * i, sw + 8 * i);
    uint32_t mx = sw[0];                         // scales are >= 0: fp16 bits order them
#pragma unroll
    for (int i = 1; i < QD / 2; ++i) mx = __vmaxu2(mx, sw[i]);
    mx = max(mx & 0xffffu, mx >> 16);
    mx = max(mx, __shfl_xor_sync(kFullMask, mx, 1));
    mx = max(mx, __shfl_xor_sync(kFullMask, mx, 2));
    const int ex = max(static_cast<int>(mx >> 10), 1) - 15;    // subnormal: -14
    const float up = __int_as_float((127 + ex) << 23);
    // 2^-ex as fp16 (2^-16 .. 2^14; below 2^-14 a subnormal): s 2^-ex is exact
    // unless it falls below 2^-14, i.e. for scales under 2^-15 of the page's
    // largest, whose terms are then rounded at 2^-24 -- far below the
    // precision of the largest terms' hi / lo parts
    const unsigned dh = -ex >= -14 ? static_cast<unsigned>(15 - ex) << 10 : 1u << (24 - ex);
    const uint32_t down2 = dh | (dh << 16);
    float qf[QD];
    const uint32_t qa = smem_u32(sm.qtab + (g >> 1) * D + c * QD);
#pragma unroll
    for (int i = 0; i < QD / 4; ++i)
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(qf[4 * i]), "=f"(qf[4 * i + 1]), "=f"(qf[4 * i + 2]), "=f"(qf[4 * i + 3])
                   : "r"(qa + 16 * i));
    auto bfrag = [&](int i) -> uint32_t {
      int d0, d1;
      kpair_dims<D, BK>(0, i, d0, d1);           // dims within the group
      // (s_d0, s_d1) in one fp16 pair, times 2^-ex, widened
      const uint32_t sp = __byte_perm(sw[d0 >> 1], sw[d1 >> 1],
                                      ((d0 & 1) ? 0x0032u : 0x0010u) | ((d1 & 1) ? 0x7600u : 0x5400u));
      __half2 sd = __hmul2(*reinterpret_cast<const __half2*>(&sp),
                           *reinterpret_cast<const __half2*>(&down2));
      const float2 sf = __half22float2(sd);
      float x0, x1, l0, l1;
      mul2(qf[d0], qf[d1], sf.x, sf.y, x0, x1);
      const __half2 hi = __floats2half2_rn(x0, x1);
      const float2 hf = __half22float2(hi);
      sub2(x0, x1, hf.x, hf.y, l0, l1);
      const __half2 lo = __floats2half2_rn(l0, l1);
      const __half2 r = (g & 1) ? lo : hi;
      return *reinterpret_cast<const uint32_t*>(&r);
    };
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const uint32_t x[4] = {kpair_signed<BK>(w0, 2 * j), kpair_signed<BK>(w1, 2 * j),
                             kpair_signed<BK>(w0, 2 * j + 1), kpair_signed<BK>(w1, 2 * j + 1)};
      mma_16816(a, x, bfrag(2 * j), bfrag(2 * j + 1));
    }
    sc0 = (a[0] + a[1]) * up;
    sc1 = (a[2] + a[3]) * up;
  };
  // p s -> B fragments of the V-side MMA (via two 8x8 transposes); l, zacc.
  // With `guard`, a token with p = 0 (masked) contributes nothing even if its
  // slot holds a non-finite scale or zero.
  auto pfrag = [&](float p0, float p1, float ps0, float ps1, float2 v0, float2 v1, bool guard,
                   uint32_t& pb0, uint32_t& pb1) {
    float z0 = v0.y, z1 = v1.y;
    if (guard) {
      if (!(p0 > 0.f)) { ps0 = 0.f; z0 = 0.f; }
      if (!(p1 > 0.f)) { ps1 = 0.f; z1 = 0.f; }
    }
    zacc = __fmaf_rn(p0, z0, zacc);
    zacc = __fmaf_rn(p1, z1, zacc);
    l += p0 + p1;
    pb0 = movm_trans(hilo_pair(ps0));
    pb1 = movm_trans(hilo_pair(ps1));
  };
  // values: token pairs (2c, 2c+1) and (2c+8, 2c+9), dims [g D/8, (g+1) D/8)
  auto pv = [&](uint32_t st, uint32_t pb0, uint32_t pb1) {
    uint32_t a0[VWORDS], a1[VWORDS], b0[VWORDS], b1[VWORDS];
    lds_u32<VSLICE>(st + voff, a0);
    lds_u32<VSLICE>(st + voff + VB, a1);
    lds_u32<VSLICE>(st + voff + 8 * VB, b0);
    lds_u32<VSLICE>(st + voff + 9 * VB, b1);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const uint32_t x[4] = {vpair<BV>(a0, a1, 2 * j), vpair<BV>(a0, a1, 2 * j + 1),
                             vpair<BV>(b0, b1, 2 * j), vpair<BV>(b0, b1, 2 * j + 1)};
      mma_16816(oacc[j], x, pb0, pb1);
    }
  };
  // Lazy running maximum (log2 units): m is raised only when a score exceeds
  // it by more than kMaxSlack, so p = 2^(score - m) <= 2^kMaxSlack; any m
  // gives the same o = acc / l once acc, l and zacc are rescaled with it.
  // thr = m + kMaxSlack in scaled units.
  const float slack = kMaxSlack / iscl;
  float thr = -CUDART_INF_F;
  // raise the running maximum of head c to cover m_loc (scaled units)
  auto rescale = [&](float m_loc) {
    const float mnew = fmaxf(m_s, warp_max_group(m_loc));
    const bool grow = mnew > m_s;
    const float alpha = grow ? ex2((m_s - mnew) * iscl) : 1.f;
    l *= alpha;
    zacc *= alpha;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      oacc[j][0] *= alpha; oacc[j][1] *= alpha; oacc[j][2] *= alpha; oacc[j][3] *= alpha;
    }
    if (grow) {
      m_s = mnew;
      mneg = -mnew * iscl;
      thr = mnew + slack;
    }
  };
  // tokens a masked round leaves out: at or beyond lq (only the last page of a
  // sequence has any) and, in LogQuant mode, the members of B (lq = len then)
  const int lq_w = LQ ? p.lq_w : 0, lq_a = LQ ? p.lq_a : 0;
  auto excluded = [&](int t) -> bool {
    return t >= lq || (LQ && lq_member32(t, lq, lq_w, lq_a));
  };
  // one round: pages A (stage at sta) and, if has_b, B (the next stage); mask
  // applies excluded() to its tokens
  auto round = [&](uint32_t sta, bool has_b, bool mask, int tok_a) {
    const uint32_t stb = sta + stage_bytes;
    float sa0, sa1, sb0 = -CUDART_INF_F, sb1 = -CUDART_INF_F;
    if constexpr (KPC2) {
      scores_kpc2(sta, sa0, sa1);
      if (has_b) scores_kpc2(stb, sb0, sb1);
    } else if constexpr (KPC4) {
      scores_kpc4(sta, sa0, sa1);
      if (has_b) scores_kpc4(stb, sb0, sb1);
    } else if constexpr (KPC) {
      scores_kpc(sta, sa0, sa1);
      if (has_b) scores_kpc(stb, sb0, sb1);
    } else {
      scores(sta, sa0, sa1);
      if (has_b) scores(stb, sb0, sb1);
    }
    if (mask) {
      const int tok_b = tok_a + kDecodeWarps * kPage;
      if (excluded(tok_a + g)) sa0 = -CUDART_INF_F;
      if (excluded(tok_a + g + 8)) sa1 = -CUDART_INF_F;
      if (excluded(tok_b + g)) sb0 = -CUDART_INF_F;
      if (excluded(tok_b + g + 8)) sb1 = -CUDART_INF_F;
    }
    const float m_loc = fmaxf(fmaxf(sa0, sa1), fmaxf(sb0, sb1));
    const float2 va0 = lds_half2(sta + VSZ + 4 * g), va1 = lds_half2(sta + VSZ + 4 * g + 32);
    float2 vb0 = make_float2(0.f, 0.f), vb1 = vb0;
    if (has_b) {
      vb0 = lds_half2(stb + VSZ + 4 * g);
      vb1 = lds_half2(stb + VSZ + 4 * g + 32);
    }
    float p[4], ps[4];
    auto probs = [&]() {
      p[0] = ex2(__fmaf_rn(sa0, iscl, mneg));
      p[1] = ex2(__fmaf_rn(sa1, iscl, mneg));
      p[2] = ex2(__fmaf_rn(sb0, iscl, mneg));
      p[3] = ex2(__fmaf_rn(sb1, iscl, mneg));
      ps[0] = p[0] * va0.x;
      ps[1] = p[1] * va1.x;
      ps[2] = p[2] * vb0.x;
      ps[3] = p[3] * vb1.x;
    };
    probs();
    // one vote: a score past the slack raises the maximum, and p s must fit
    // fp16 (a very large value scale takes the exact maximum, p <= 1, p s <= s);
    // either way this round's p are taken again with the raised maximum
    const bool slow = m_loc > thr || fmaxf(fmaxf(ps[0], ps[1]), fmaxf(ps[2], ps[3])) > kMaxPS;
    if (__any_sync(kFullMask, slow)) {
      rescale(m_loc);
      probs();
    }
    uint32_t pa0, pa1, pb0, pb1;
    pfrag(p[0], p[1], ps[0], ps[1], va0, va1, mask, pa0, pa1);
    if (has_b) pfrag(p[2], p[3], ps[2], ps[3], vb0, vb1, mask, pb0, pb1);
    pv(sta, pa0, pa1);
    if (has_b) pv(stb, pb0, pb1);
  };

  const int lq_from = LQ ? lq_lo(lq, lq_w, lq_a) : 0;
  // the last page of the sequence is partial unless lq is a multiple of 16
  const bool last_partial = (lq % kPage) != 0 && nk > 0 &&
                            first + kDecodeWarps * (nk - 1) == npages - 1;
  // the main loop covers full pages without the new token (kpatch, when set,
  // is this warp's last page); the final round takes the rest
  const int nfull = nk - ((last_partial || kpatch >= 0) ? 1 : 0);

  if (p.wait_log2 < kWaitLimitLog2)
    for (int kk = 0; kk < nk && kk < NST; ++kk) issue(true, kk, pid_of(kk));
  bool timed_out = false;
  int k = 0, sa = 0;
  unsigned ph = 0;
  // full rounds: RP full pages each
  constexpr int RP = kDecodeRoundPages;
  for (; k + RP <= nfull;) {
    bool ok;
    if constexpr (RP == 2) {
      ok = mbar_wait2_warp(bars + sa, ph, sm.wait_log2);
    } else {
      int lim;
      asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(lim) : "r"(smem_u32(sm.wait_log2)));
      ok = __all_sync(kFullMask, mbar_wait_bounded(bars + sa, ph, lim));
    }
    if (!ok) {
      timed_out = true;
      break;
    }
    if constexpr (LQ) {
      // pages first + 4k (, first + 4k + 4): members lie in block 0 and from
      // lq_lo() on
      const int t0 = (first + kDecodeWarps * k) * kPage;
      const int t1 = t0 + (RP == 2 ? kDecodeWarps * kPage : 0) + kPage;
      // masked rounds are rare (block 0 and the newest positions): a literal
      // flag per call gives the common unmasked round its own copy
      if (t0 < lq_w || t1 > lq_from) round(st0 + sa * stage_bytes, RP == 2, true, t0);
      else round(st0 + sa * stage_bytes, RP == 2, false, t0);
    } else {
      round(st0 + sa * stage_bytes, RP == 2, false, 0);
    }
    // refill the round's stages with pages k + NST (, k + NST + 1)
    const int pid0 = pid_of(k + NST);
    const int pid1 = RP == 2 ? pid_of(k + NST + 1) : 0;
    __syncwarp();
    issue(k + NST < nk, sa, pid0);
    if constexpr (RP == 2) issue(k + NST + 1 < nk, sa + 1, pid1);
    k += RP;
    sa += RP;
    if (sa == NST) {
      sa = 0;
      ph ^= 1u;
    }
    if (k >= 32 * (chunk + 1)) {
      ++chunk;
      pid_cur = pid_nxt;
      pid_nxt = load_chunk(chunk + 1);
    }
  }
  // the rest: at most RP pages, the last maybe partial
  if (!timed_out && k < nk) {
    const bool has_b = RP == 2 && k + 1 < nk;
    bool ok = mbar_wait_bounded(bars + sa, ph, *sm.wait_log2);
    if (has_b) ok = mbar_wait_bounded(bars + sa + 1, ph, *sm.wait_log2) && ok;
    if (!__all_sync(kFullMask, ok)) {
      timed_out = true;
    } else {
      if constexpr (!KPC) {
        if (kpatch >= 0 && (kpatch - k) >= 0 && (kpatch - k) < (has_b ? 2 : 1))
          patch_stage<D, BK, BV>(st0 + (sa + kpatch - k) * stage_bytes, pbuf, pslot);
      }
      round(st0 + sa * stage_bytes, has_b, last_partial || LQ,
            (first + kDecodeWarps * k) * kPage);
    }
  }
  if (timed_out) {
    if (lane == 0) flag_status(p.status, KVQ_DEV_COPY_TIMEOUT);
    // drain the copies still in flight (pages k .. k + NST - 1), with the full
    // limit: none of them may land after the CTA has exited
    int s = sa;
    unsigned q = ph;
    for (int kk = k; kk < nk && kk < k + NST; ++kk) {
      (void)mbar_wait_bounded(bars + s, q);
      if (++s == NST) {
        s = 0;
        q ^= 1u;
      }
    }
  }

  // ---- key-per-channel mode without a window: the open page's bf16 rows
  //      (positions lq .. len - 1, at most 15, ring slots p % 16) join the
  //      last split's online softmax, so that no window CTA holds a slot of
  //      the wave.  Each row is rotated like the query (H k, H v; lane l holds
  //      dims [E l, E l + E)): score = sum_d qtab[c][d] (H k)_d, the same
  //      scaled units as the pages' scores; lane (g, c) adds p (H v) over its
  //      accumulator dims [g D / 8, (g + 1) D / 8), held by lanes 4 g .. 4 g + 3.
  if constexpr (KPC) {
    if (!timed_out && p.NS == p.S && split == p.S - 1) {
      constexpr int E = D / 32;
      const uint16_t* kplane = p.window + (static_cast<size_t>(b) * p.Hkv + h) * 2 * p.R * D;
      const uint16_t* vplane = kplane + static_cast<size_t>(p.R) * D;
      for (int t = lq + warp; t < len; t += kDecodeWarps) {
        const size_t row = static_cast<size_t>(t % p.R) * D + E * lane;
        float kx[E], vx[E];
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const uint32_t kw = *reinterpret_cast<const uint32_t*>(kplane + row + e);
          const uint32_t vw = *reinterpret_cast<const uint32_t*>(vplane + row + e);
          kx[e] = bf16lo(kw); kx[e + 1] = bf16hi(kw);
          vx[e] = bf16lo(vw); vx[e + 1] = bf16hi(vw);
        }
        warp_fwht<E>(kx, p.had_block);
        float a[kMaxGroup];
#pragma unroll
        for (int i = 0; i < kMaxGroup; ++i) {
          a[i] = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            float qe = sm.qtab[i * D + E * lane + e];
            if constexpr (KPC2 || KPC4) {        // the packed (hi, lo) pair of e q''
              const uint32_t hl = __float_as_uint(qe);
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hl));
              qe = f.x + f.y;
            }
            a[i] = __fmaf_rn(qe, kx[e], a[i]);
          }
          a[i] = warp_sum(a[i]);
        }
        const float sc = c == 0 ? a[0] : c == 1 ? a[1] : c == 2 ? a[2] : a[3];
        if (__any_sync(kFullMask, sc > thr)) rescale(sc);
        const float pr = ex2(__fmaf_rn(sc, iscl, mneg));
        if (g == 0) l += pr;
        warp_fwht<E>(vx, p.had_block);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float val = __shfl_sync(kFullMask, vx[e], (lane & ~3) + k4);
            const int m = E * k4 + e;               // dim g D / 8 + m
            oacc[m >> 1][(m & 1) * 2] = __fmaf_rn(pr, val, oacc[m >> 1][(m & 1) * 2]);
          }
        }
      }
    }
  }

  // ---- warp partial -> the merge region (the caller merges the warps)
  l = warp_sum_group(l);
  zacc = warp_sum_group(zacc);
  const float m = m_s == -CUDART_INF_F ? -CUDART_INF_F : m_s * iscl;
  __syncthreads();  // every warp is done with its stage buffers
  float* macc = sm.merge;                                    // [warps][kMaxGroup][D]
  float* mml = macc + kDecodeWarps * kMaxGroup * D;          // m, l: [warps][kMaxGroup] each
  float* wrow = macc + (warp * kMaxGroup + c) * D;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    wrow[g * (D / 8) + 2 * j] = oacc[j][0] + oacc[j][1] + zacc;
    wrow[g * (D / 8) + 2 * j + 1] = oacc[j][2] + oacc[j][3] + zacc;
  }
  if (g == 0) {
    mml[warp * kMaxGroup + c] = m;
    mml[kDecodeWarps * kMaxGroup + warp * kMaxGroup + c] = l;
  }
}

// ---------------------------------------------- bf16 rows: window, reserve
// Attention of the G query heads over nw bf16 rows (K row t at krow(t), V row
// t at vrow(t)), written as an unrotated partial (m, l, acc) into `part`.  The
// rows may come in any order (attention is order-free).  Lane l holds dims
// [E l, E l + E) of a row; each warp keeps UNROLL rows in flight.
//   1. scores: warp w takes rows w, w + 4, ...; each lane forms its dims'
//      partial dot products with the G query heads, and one transpose-reduce
//      (6 shuffles) leaves head (2 [l >= 16] + [l & 8]) summed in each group of
//      8 lanes;
//   2. warp i: maximum and sum of head i, p = 2^(s - m) in place;
//   3. values: warp w takes the same rows, accumulates p v for every head
//      in registers; the warps' sums meet in shared memory.
// sc: [kMaxGroup][ldsc] floats of shared memory (ldsc >= nw).
template <int D, typename KRow, typename VRow>
__device__ void attend_rows(const DecodeParams& p, const Smem& sm, int nw, float* sc, int ldsc,
                            KRow krow, VRow vrow, float* part) {
  constexpr int E = D / 32;
  constexpr int RW = E / 2;     // packed bf16 words of a row per lane
  constexpr int UNROLL = 16;    // rows in flight per warp
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto load_row = [&](const uint16_t* row, uint32_t (&w)[RW]) {
    const uint16_t* src = row + E * lane;
    if constexpr (E == 4) {
      const uint2 x = *reinterpret_cast<const uint2*>(src);
      w[0] = x.x;
      w[1] = x.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(src);
    }
  };
  auto unpack = [&](const uint32_t (&w)[RW], float (&x)[E]) {
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      x[2 * i] = bf16lo(w[i]);
      x[2 * i + 1] = bf16hi(w[i]);
    }
  };
  float qf[kMaxGroup][E];
#pragma unroll
  for (int i = 0; i < kMaxGroup; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) qf[i][e] = sm.qtab[i * D + E * lane + e];
  const bool up = lane & 16, u8 = lane & 8;
  const int hsel = (up ? 2 : 0) + (u8 ? 1 : 0);

  // ---- 1. scores
  for (int t0 = warp; t0 < nw; t0 += kDecodeWarps * UNROLL) {
    uint32_t raw[UNROLL][RW];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int t = t0 + kDecodeWarps * u;
      if (t < nw) load_row(krow(t), raw[u]);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int t = t0 + kDecodeWarps * u;
      if (t >= nw) break;                       // warp-uniform
      float x[E];
      unpack(raw[u], x);
      float a[kMaxGroup];
#pragma unroll
      for (int i = 0; i < kMaxGroup; ++i) {
        a[i] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) a[i] = __fmaf_rn(qf[i][e], x[e], a[i]);
      }
      // lanes < 16 keep heads 0, 1 and lanes >= 16 heads 2, 3; then bit 3
      // picks one of the two; then a sum over the 8 lanes
      const float r0 = __shfl_xor_sync(kFullMask, up ? a[0] : a[2], 16);
      const float r1 = __shfl_xor_sync(kFullMask, up ? a[1] : a[3], 16);
      const float k0 = (up ? a[2] : a[0]) + r0, k1 = (up ? a[3] : a[1]) + r1;
      float vv = (u8 ? k1 : k0) + __shfl_xor_sync(kFullMask, u8 ? k0 : k1, 8);
      vv += __shfl_xor_sync(kFullMask, vv, 4);
      vv += __shfl_xor_sync(kFullMask, vv, 2);
      vv += __shfl_xor_sync(kFullMask, vv, 1);
      if ((lane & 7) == 0) sc[hsel * ldsc + t] = vv;
    }
  }
  __syncthreads();
  // ---- 2. softmax statistics of query head i (warp i)
  if (warp < p.G) {
    float mm = -CUDART_INF_F;
    for (int t = lane; t < nw; t += 32) mm = fmaxf(mm, sc[warp * ldsc + t]);
    mm = warp_max(mm);
    float ll = 0.f;
    for (int t = lane; t < nw; t += 32) {
      const float e = ex2(sc[warp * ldsc + t] - mm);
      sc[warp * ldsc + t] = e;
      ll += e;
    }
    ll = warp_sum(ll);
    if (lane == 0) {
      part_m<D>(part)[warp] = nw > 0 ? mm : -CUDART_INF_F;
      part_l<D>(part)[warp] = ll;
    }
  }
  __syncthreads();
  // ---- 3. values
  float acc[kMaxGroup][E];
#pragma unroll
  for (int i = 0; i < kMaxGroup; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
  for (int t0 = warp; t0 < nw; t0 += kDecodeWarps * UNROLL) {
    uint32_t raw[UNROLL][RW];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int t = t0 + kDecodeWarps * u;
      if (t < nw) load_row(vrow(t), raw[u]);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int t = t0 + kDecodeWarps * u;
      if (t >= nw) break;
      float x[E];
      unpack(raw[u], x);
#pragma unroll
      for (int i = 0; i < kMaxGroup; ++i) {
        const float pi = i < p.G ? sc[i * ldsc + t] : 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = __fmaf_rn(pi, x[e], acc[i][e]);
      }
    }
  }
  __syncthreads();  // every warp is done with the scores (the merge region shares them)
  float* macc = sm.merge;                       // [warps][kMaxGroup][D]
#pragma unroll
  for (int i = 0; i < kMaxGroup; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) macc[(warp * kMaxGroup + i) * D + E * lane + e] = acc[i][e];
  __syncthreads();
  for (int idx = tid; idx < kMaxGroup * D; idx += kThreads) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) sum += macc[w * kMaxGroup * D + idx];
    part[idx] = sum;                            // part_acc<D>(part, i)[d], idx = i D + d
  }
}

// Shared memory of the window split: scores [kMaxGroup][R] (128-byte
// aligned), then up to kWinChunk rows of the ring [rows][D] bf16.
constexpr int kWinChunk = 128;
__host__ __device__ constexpr size_t win_score_bytes(int R) {
  return (static_cast<size_t>(kMaxGroup) * R * 4 + 127) / 128 * 128;
}
__host__ __device__ constexpr size_t win_bytes(int R, int d) {
  return win_score_bytes(R) + static_cast<size_t>(R < kWinChunk ? R : kWinChunk) * d * 2;
}

// The bf16 window of (b, h): tokens at positions lq .. len - 1, in ring slots
// p % R.  The valid slots are always the prefix [0, len - lq) of the ring (all
// R of them once the sequence is longer than the window), and attention is
// order-free, so the slots are taken in storage order: chunks of up to
// kWinChunk rows are staged in shared memory by one bulk copy each (the kernel
// start has prefetched the window into L2), K for the scores, then V.  The
// decode step's newest token comes from k_new / v_new: its slot is being
// rewritten by this launch.  Lane l holds dims [E l, E l + E) of a row; warp w
// takes rows w, w + 4, ... of each chunk.
template <int D>
__device__ void window_split(const DecodeParams& p, const Smem& sm, int b, int h, int len, int lq,
                             float* part) {
  constexpr int E = D / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nw = len - lq;
  const int R = p.R;
  // the key-per-channel ring (R + 16 rows) holds positions lq .. len - 1 at
  // slots p % R: a run of nw slots from lq % R that may wrap around the end
  const int s0 = p.kpc ? lq % R : 0;
  const uint16_t* kring = p.window + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + 0) * R * D;
  const uint16_t* vring = kring + static_cast<size_t>(R) * D;
  const int snew = (p.step && nw > 0) ? (len - 1) % R : -1;
  const uint16_t* knew = p.step ? p.k_new + (static_cast<size_t>(b) * p.Hkv + h) * D : nullptr;
  const uint16_t* vnew = p.step ? p.v_new + (static_cast<size_t>(b) * p.Hkv + h) * D : nullptr;
  float* sc = reinterpret_cast<float*>(sm.area);                       // [kMaxGroup][R]
  uint16_t* buf = reinterpret_cast<uint16_t*>(sm.area + win_score_bytes(R));  // [chunk][D]
  uint64_t* bar = sm.bars;              // this CTA has no page ring: its first barrier
  unsigned ph = 0;
  // rows [c0, c0 + n) of a ring plane into buf (every thread waits)
  auto stage = [&](const uint16_t* plane, int c0, int n) {
    __syncthreads();                    // everyone is done with buf
    if (tid == 0) {
      mbar_expect_tx(bar, static_cast<unsigned>(n) * D * 2);
      const int first = (s0 + c0) % R;
      const int n1 = min(n, R - first); // rows before the ring's end
      bulk_g2s(buf, plane + static_cast<size_t>(first) * D, static_cast<unsigned>(n1) * D * 2, bar);
      if (n1 < n)
        bulk_g2s(buf + static_cast<size_t>(n1) * D, plane, static_cast<unsigned>(n - n1) * D * 2,
                 bar);
    }
    if (!mbar_wait_bounded(bar, ph)) {
      if (tid == 0) flag_status(p.status, KVQ_DEV_COPY_TIMEOUT);
      (void)mbar_wait_bounded(bar, ph); // the copy must land before buf is reused
    }
    ph ^= 1u;
  };
  // this lane's E values of slot t (chunk base c0), as floats
  auto row = [&](const uint16_t* fresh, int t, int c0, float (&x)[E]) {
    uint32_t w[E / 2];
    if (t == snew) {
      const uint16_t* src = fresh + E * lane;
#pragma unroll
      for (int i = 0; i < E / 2; ++i) w[i] = *reinterpret_cast<const uint32_t*>(src + 2 * i);
    } else {
      const uint32_t a = smem_u32(buf + static_cast<size_t>(t - c0) * D + E * lane);
      if constexpr (E == 4) {
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(a));
      } else {
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[0]) : "r"(a));
      }
    }
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      x[2 * i] = bf16lo(w[i]);
      x[2 * i + 1] = bf16hi(w[i]);
    }
  };
  float qf[kMaxGroup][E];
#pragma unroll
  for (int i = 0; i < kMaxGroup; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) qf[i][e] = sm.qtab[i * D + E * lane + e];
  const bool up = lane & 16, u8 = lane & 8;
  const int hsel = (up ? 2 : 0) + (u8 ? 1 : 0);

  // ---- 1. scores: each lane forms its dims' partial dot products with the G
  //      query heads; one transpose-reduce (6 shuffles) leaves head (2 [l >=
  //      16] + [l & 8]) summed in each group of 8 lanes
  for (int c0 = 0; c0 < nw; c0 += kWinChunk) {
    const int n = min(kWinChunk, nw - c0);
    stage(kring, c0, n);
    for (int t = c0 + warp; t < c0 + n; t += kDecodeWarps) {
      float x[E];
      row(knew, t, c0, x);
      float a[kMaxGroup];
#pragma unroll
      for (int i = 0; i < kMaxGroup; ++i) {
        a[i] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) a[i] = __fmaf_rn(qf[i][e], x[e], a[i]);
      }
      const float r0 = __shfl_xor_sync(kFullMask, up ? a[0] : a[2], 16);
      const float r1 = __shfl_xor_sync(kFullMask, up ? a[1] : a[3], 16);
      const float k0 = (up ? a[2] : a[0]) + r0, k1 = (up ? a[3] : a[1]) + r1;
      float vv = (u8 ? k1 : k0) + __shfl_xor_sync(kFullMask, u8 ? k0 : k1, 8);
      vv += __shfl_xor_sync(kFullMask, vv, 4);
      vv += __shfl_xor_sync(kFullMask, vv, 2);
      vv += __shfl_xor_sync(kFullMask, vv, 1);
      if ((lane & 7) == 0) sc[hsel * R + t] = vv;
    }
  }
  __syncthreads();
  // ---- 2. softmax statistics of query head i (warp i)
  if (warp < p.G) {
    float mm = -CUDART_INF_F;
    for (int t = lane; t < nw; t += 32) mm = fmaxf(mm, sc[warp * R + t]);
    mm = warp_max(mm);
    float ll = 0.f;
    for (int t = lane; t < nw; t += 32) {
      const float e = ex2(sc[warp * R + t] - mm);
      sc[warp * R + t] = e;
      ll += e;
    }
    ll = warp_sum(ll);
    if (lane == 0) {
      part_m<D>(part)[warp] = nw > 0 ? mm : -CUDART_INF_F;
      part_l<D>(part)[warp] = ll;
    }
  }
  // ---- 3. values: p v for every head in registers; the warps' sums meet in
  //      shared memory (stage() begins with the barrier that orders phase 2)
  float acc[kMaxGroup][E];
#pragma unroll
  for (int i = 0; i < kMaxGroup; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
  for (int c0 = 0; c0 < nw; c0 += kWinChunk) {
    const int n = min(kWinChunk, nw - c0);
    stage(vring, c0, n);
    for (int t = c0 + warp; t < c0 + n; t += kDecodeWarps) {
      float x[E];
      row(vnew, t, c0, x);
#pragma unroll
      for (int i = 0; i < kMaxGroup; ++i) {
        const float pi = i < p.G ? sc[i * R + t] : 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = __fmaf_rn(pi, x[e], acc[i][e]);
      }
    }
  }
  __syncthreads();
  float* macc = sm.merge;                       // [warps][kMaxGroup][D]
#pragma unroll
  for (int i = 0; i < kMaxGroup; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) macc[(warp * kMaxGroup + i) * D + E * lane + e] = acc[i][e];
  __syncthreads();
  for (int idx = tid; idx < kMaxGroup * D; idx += kThreads) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) sum += macc[w * kMaxGroup * D + idx];
    part[idx] = sum;                            // part_acc<D>(part, i)[d], idx = i D + d
  }
  // decode step on a sequence no longer than the window: no token leaves the
  // ring, so nobody else writes the new token into it
  if (p.step && lq == 0 && nw > 0) {
    uint16_t* kslot = const_cast<uint16_t*>(kring) + static_cast<size_t>((len - 1) % R) * D;
    uint16_t* vslot = kslot + static_cast<size_t>(R) * D;
    for (int d = tid; d < D; d += kThreads) {
      kslot[d] = knew[d];
      vslot[d] = vnew[d];
    }
  }
}

// Reserve split r of nr (LogQuant mode) of (b, h) at length len.  In a decode
// step, split 0 carries out the halving, if the token fills B to 3W (the block
// thinned for the first time moves from the ring to its level buffer; the
// first halving moves block 0 too), and writes the token's bf16 rows into the
// ring.  Then each split lists the rows of its share of B's members in shared
// memory (any order) and attends over them.
template <int D>
__device__ void reserve_split(const DecodeParams& p, const Smem& sm, int b, int h, int len,
                              int r, int nr, float* part) {
  const int tid = threadIdx.x;
  const int w = p.lq_w, a = p.lq_a, half = w / 2;
  const int ldsc = 3 * w;                       // |B| <= 3W
  float* sc = reinterpret_cast<float*>(sm.area);           // [kMaxGroup][3W]
  int* list = reinterpret_cast<int*>(sc + kMaxGroup * ldsc); // [3W] row numbers
  int* count = reinterpret_cast<int*>(sm.flag);
  uint16_t* kplane = const_cast<uint16_t*>(p.window) +
                     ((static_cast<size_t>(b) * p.Hkv + h) * 2) * p.lq_rows * D;
  uint16_t* vplane = kplane + static_cast<size_t>(p.lq_rows) * D;
  constexpr int C = D / 8;                      // uint4 chunks per row
  // a decode step's halving (block 1 + k0, and block 0 at the first one) and
  // new token: reserve CTA 0 writes them for the later steps, and every reserve
  // CTA reads those rows where they were before this step (the ring, k_new /
  // v_new), so that none depends on another's writes
  const int k0 = p.step && len > 0 ? lq_halvings(len - 1, w) : 0;
  const int k1 = p.step && len > 0 ? lq_halvings(len, w) : 0;
  if (p.step && len > 0 && r == 0) {
    if (k1 > k0) {                              // one halving: block 1 + k0 (and block 0)
      for (int pass = 0; pass < (k0 == 0 ? 2 : 1); ++pass) {
        const int bb = pass ? 0 : 1 + k0;
        const int level = bb == 0 ? a : bb % a;
        for (int idx = tid; idx < 2 * half * C; idx += kThreads) {
          const int kv = idx / (half * C), r = idx - kv * half * C;
          const int v = r / C, ci = r - v * C;
          const int q = bb * w + 2 * v;         // older than this step's token
          uint16_t* plane = kv ? vplane : kplane;
          const uint4 x = reinterpret_cast<const uint4*>(plane + static_cast<size_t>(q % (3 * w)) * D)[ci];
          reinterpret_cast<uint4*>(plane + static_cast<size_t>(3 * w + level * half + v) * D)[ci] = x;
        }
      }
    }
    // the new token: a member, newer than (k + 1) W: its ring row
    const int rnew = (len - 1) % (3 * w);
    const uint16_t* knew = p.k_new + (static_cast<size_t>(b) * p.Hkv + h) * D;
    const uint16_t* vnew = p.v_new + (static_cast<size_t>(b) * p.Hkv + h) * D;
    for (int idx = tid; idx < 2 * C; idx += kThreads) {
      const int kv = idx / C, ci = idx - kv * C;
      reinterpret_cast<uint4*>((kv ? vplane : kplane) + static_cast<size_t>(rnew) * D)[ci] =
          reinterpret_cast<const uint4*>(kv ? vnew : knew)[ci];
    }
  }
  if (tid == 0) *count = 0;
  __syncthreads();
  // member list: block 0 and the positions from lq_lo on, candidates t with
  // t mod nr = r for reserve CTA r; the row each is read from (-1: the new
  // token, read from k_new / v_new)
  const int lo = lq_lo(len, w, a);
  const int nb0 = min(w, len);
  const int ncand = nb0 + max(0, len - max(lo, nb0));
  const int moved = k1 > k0 ? 1 + k0 : -1;      // block moved by this step's halving
  for (int t = r + nr * tid; t < ncand; t += nr * kThreads) {
    const int pos = t < nb0 ? t : max(lo, nb0) + (t - nb0);
    if (!lq_member32(pos, len, w, a)) continue;
    int row = lq_row32(pos, len, w, a);
    if (p.step) {
      if (pos == len - 1) row = -1;
      else if (moved >= 0 && ((pos >> a) == moved || (k0 == 0 && (pos >> a) == 0)))
        row = pos % (3 * w);                    // still in the ring before this step
    }
    list[atomicAdd(count, 1)] = row;
  }
  __syncthreads();
  const int nm = *count;
  const uint16_t* knew = p.step ? p.k_new + (static_cast<size_t>(b) * p.Hkv + h) * D : nullptr;
  const uint16_t* vnew = p.step ? p.v_new + (static_cast<size_t>(b) * p.Hkv + h) * D : nullptr;
  attend_rows<D>(
      p, sm, nm, sc, ldsc,
      [&](int t) { return list[t] < 0 ? knew : kplane + static_cast<size_t>(list[t]) * D; },
      [&](int t) { return list[t] < 0 ? vnew : vplane + static_cast<size_t>(list[t]) * D; }, part);
}

// E consecutive floats (E = 4 or 2; 16- or 8-byte aligned) bypassing L1.
template <int E>
__device__ __forceinline__ void ldcg_vec(const float* ptr, float (&v)[E]) {
  if constexpr (E == 4) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(ptr));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(ptr));
    v[0] = x.x; v[1] = x.y;
  }
}

// Ticket mode.  Warp i merges query head i of (b, h) over its NS global
// partials (L2-resident: this launch wrote them):
//   1. every partial's m and l in one pass (lane k holds splits k + 32 j, all
//      loads in flight at once), the maximum, the weights 2^(m_s - M) -- kept
//      in shared memory (`wsm`, the free stage area) for the next step -- and L;
//   2. the weighted sum of the quantized splits' rotated accumulators (E dims
//      per lane, kCombineRows rows in flight per lane);
//   3. the inverse rotation x = H u / n, the window or reserve splits'
//      accumulators (already in the model's basis), and o.
constexpr int kMaxNS = kMaxSplits + 4;      // splits + window / reserve CTAs
constexpr int kCombineRows = 16;
template <int D>
__device__ void combine_global(const DecodeParams& p, const Smem& sm, int b, int h,
                               const float* parts) {
  constexpr int E = D / 32;
  constexpr int PS = kMaxGroup * (D + 2);   // floats per partial
  constexpr int UN = kCombineRows;
  constexpr int NJ = (kMaxNS + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= p.G) return;
  const int i = warp, NS = p.NS, nq = p.S;
  float* wsm = reinterpret_cast<float*>(sm.area) + i * kMaxNS;
  float ms[NJ], ls[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int s = lane + 32 * j;
    ms[j] = -CUDART_INF_F;
    ls[j] = 0.f;
    if (s < NS) {
      ms[j] = __ldcg(part_m<D>(parts + s * PS) + i);
      ls[j] = __ldcg(part_l<D>(parts + s * PS) + i);
    }
  }
  float mm = ms[0];
#pragma unroll
  for (int j = 1; j < NJ; ++j) mm = fmaxf(mm, ms[j]);
  mm = warp_max(mm);
  float ll = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int s = lane + 32 * j;
    if (s < NS) {
      const float w = ms[j] == -CUDART_INF_F ? 0.f : exp2f(ms[j] - mm);
      ll = __fmaf_rn(w, ls[j], ll);
      wsm[s] = w;
    }
  }
  ll = warp_sum(ll);
  __syncwarp();
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int k0 = 0; k0 < nq; k0 += UN) {
    float rows[UN][E];
#pragma unroll
    for (int k = 0; k < UN; ++k) {
      if (k0 + k < nq) {
        ldcg_vec<E>(part_acc<D>(parts + (k0 + k) * PS, i) + E * lane, rows[k]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) rows[k][e] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < UN; ++k) {
      const float wv = k0 + k < nq ? wsm[k0 + k] : 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(wv, rows[k][e], acc[e]);
    }
  }
  warp_fwht<E>(acc, p.had_block);
  const float inv_nb = 1.f / static_cast<float>(p.had_block);
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] *= inv_nb;
  // the unrotated partials (window, reserve) after the quantized ones
  for (int s = nq; s < NS; ++s) {
    const float ws = wsm[s];
    if (ws == 0.f) continue;
    float row[E];
    ldcg_vec<E>(part_acc<D>(parts + s * PS, i) + E * lane, row);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(ws, row[e], acc[e]);
  }
  float* o = p.o + (static_cast<size_t>(b) * p.Hq + h * p.G + i) * D + E * lane;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = ll > 0.f ? acc[e] / ll : 0.f;
}

// ---------------------------------------------------------- cluster merge --
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
// Cluster mode, CTA 0 after the cluster barrier: warp i merges query head i
// of (b, h) over the NS partials in rbuf (partial s from CTA rank s), as
// combine_global; a single split's own partial is cpart.
template <int D>
__device__ void combine_cluster(const DecodeParams& p, const Smem& sm, int b, int h) {
  constexpr int E = D / 32;
  constexpr int PS = kMaxGroup * (D + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= p.G) return;
  const int i = warp, NS = p.NS, nq = p.S;
  const float* rb = NS > 1 ? rbuf<D>(sm) : sm.cpart;
  float ms = -CUDART_INF_F, ls = 0.f;
  if (lane < NS) {
    ms = part_m<D>(rb + lane * PS)[i];
    ls = part_l<D>(rb + lane * PS)[i];
  }
  const float mm = warp_max(ms);
  const float w = ms == -CUDART_INF_F ? 0.f : exp2f(ms - mm);
  const float ll = warp_sum(w * ls);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxCluster; ++s) {
    const float ws = __shfl_sync(kFullMask, w, s);
    if (s < nq) {
      const float* row = part_acc<D>(rb + s * PS, i) + E * lane;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(ws, row[e], acc[e]);
    }
  }
  warp_fwht<E>(acc, p.had_block);
  const float inv_nb = 1.f / static_cast<float>(p.had_block);
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] *= inv_nb;
  for (int s = nq; s < NS; ++s) {           // the unrotated partials
    const float ws = __shfl_sync(kFullMask, w, s);
    const float* row = part_acc<D>(rb + s * PS, i) + E * lane;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(ws, row[e], acc[e]);
  }
  float* o = p.o + (static_cast<size_t>(b) * p.Hq + h * p.G + i) * D + E * lane;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = ll > 0.f ? acc[e] / ll : 0.f;
}

// Stores this CTA's partial (cpart) into slot `rank` of CTA 0's rbuf.
template <int D>
__device__ __forceinline__ void push_partial(const Smem& sm, uint32_t rank) {
  constexpr int PS = kMaxGroup * (D + 2);
  static_assert(PS % 4 == 0, "partials move as float4");
  const uint32_t dst = dsmem_addr(rbuf<D>(sm) + rank * PS, 0);
  const float4* src = reinterpret_cast<const float4*>(sm.cpart);
  for (int k = threadIdx.x; k < PS / 4; k += kThreads) {
    const float4 x = src[k];
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 16 * k),
                 "f"(x.x), "f"(x.y), "f"(x.z), "f"(x.w)
                 : "memory");
  }
}

// -------------------------------------------------------------- the kernel --
// MODE: token-wise, LogQuant or key-per-channel, each its own instantiation,
// so that the token-wise kernel's code is untouched by the other modes.
template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, kDecodeMinBlocks) decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const Smem sm = carve<D>(smem_raw, rbuf_ctas(p.cluster, p.NS));
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;

  grid_launch_dependents();

  // The query, page-id and length loads go out first: the page copies issued
  // next fill the memory system for microseconds, and a load queued behind
  // them would stall the CTA for as long.  Under programmatic dependent launch
  // the query and the new token are loaded after the wait instead.
  float qv[D / 32];
  uint32_t tok[D / 32];                 // decode step: this lane's part of the new token
  if (!p.overlap) {
    load_query<D>(p, b, h, qv);
    if (p.step && split < p.S) load_new_token<D>(p, b, h, tok);
  }
  const int chunk0 = split < p.S ? load_page_chunk0(p, b, split * p.pages_per_split) : 0;
  int len = static_cast<int>(ldg_nc_u32(p.seq_lens + b));
  if (len < p.step || len > p.max_pages * kPage) {   // a step appends one token: len >= 1
    if (tid == 0) flag_status(p.status, KVQ_DEV_BAD_LENGTH);
    len = 0;
  }
  // quantized prefix: the tokens before the window, or (key-per-channel, a
  // ring of R + 16 rows) the pages that lie wholly before the last R tokens
  const int lq = MODE == kModeKeyChannel ? kPage * (max(0, len - (p.R - kPage)) / kPage)
                 : p.R                   ? max(0, len - p.R)
                                         : len;
  const bool is_window = split >= p.S;

  if (tid == 0) {
    for (int i = 0; i < kDecodeWarps * kDecodeStages; ++i) mbar_init(sm.bars + i, 1);
    *sm.bad = 0;
    *sm.wait_log2 = p.wait_log2;
    mbar_init_fence();
  }
  __syncthreads();

  if (MODE == kModeLogQuant && is_window) {
    // the reserve's two planes of (b, h) are contiguous: one bulk prefetch into
    // L2 each, before the wait (a hint, as for the window), so that the member
    // rows the attention gathers are L2 hits when it starts
    if (tid == 0 && len > 0) {
      const uint16_t* kplane = p.window + (static_cast<size_t>(b) * p.Hkv + h) * 2 * p.lq_rows * D;
      const uint32_t bytes = static_cast<uint32_t>(p.lq_rows) * D * 2;
      l2_prefetch_bulk(kplane, bytes);
      l2_prefetch_bulk(kplane + static_cast<size_t>(p.lq_rows) * D, bytes);
    }
    grid_wait();
    if (p.overlap) load_query<D>(p, b, h, qv);
    query_window_prologue<D>(p, sm, qv);
    reserve_split<D>(p, sm, b, h, len, split - p.S, p.NS - p.S, sm.cpart);
  } else if (is_window) {
    // the window's valid slots are a prefix of the ring (all R of them once
    // the sequence is longer than the window): one bulk prefetch into L2 each
    // for K and V, before the wait (a hint; L2 is coherent with the writes
    // of the previous kernel)
    if (tid == 0 && len > 0) {
      // (the key-per-channel ring's run may wrap: the whole ring)
      const int nw = MODE == kModeKeyChannel ? p.R : len - lq;
      const uint16_t* kring = p.window + (static_cast<size_t>(b) * p.Hkv + h) * 2 * p.R * D;
      const uint32_t bytes = static_cast<uint32_t>(nw) * D * 2;
      l2_prefetch_bulk(kring, bytes);
      l2_prefetch_bulk(kring + static_cast<size_t>(p.R) * D, bytes);
    }
    grid_wait();
    if (p.overlap) load_query<D>(p, b, h, qv);
    query_window_prologue<D>(p, sm, qv);
    window_split<D>(p, sm, b, h, len, lq, sm.cpart);
  } else {
    const int bk = p.geom.bits[h][0], bv = p.geom.bits[h][1];
    switch (bk * 16 + bv) {
      case 0x22: quant_split<D, 2, 2, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x24: quant_split<D, 2, 4, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x28: quant_split<D, 2, 8, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x42: quant_split<D, 4, 2, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x44: quant_split<D, 4, 4, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x48: quant_split<D, 4, 8, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x82: quant_split<D, 8, 2, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x84: quant_split<D, 8, 4, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      case 0x88: quant_split<D, 8, 8, MODE>(p, sm, b, h, split, lq, len, qv, chunk0, tok); break;
      default: break;
    }
    __syncthreads();   // the warps' partials are in the merge region
    if (warp < p.G) merge_warps<D>(sm, warp, *reinterpret_cast<volatile int*>(sm.bad) != 0, sm.cpart);
  }
  __syncthreads();     // this CTA's partial is complete in sm.cpart

  if (p.cluster) {
    const uint32_t rank = cluster_rank();
    if (p.NS > 1) push_partial<D>(sm, rank);
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if (rank != 0) return;     // nothing reads this CTA's shared memory
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    combine_cluster<D>(p, sm, b, h);
    return;
  }
  // ticket mode: partial to global memory; the last CTA of (b, h) merges
  constexpr int PS = kMaxGroup * (D + 2);
  float* parts = p.partials + (static_cast<size_t>(b) * p.Hkv + h) * p.NS * PS;
  float* part = parts + static_cast<size_t>(split) * PS;
  for (int k = tid; k < PS; k += kThreads) part[k] = sm.cpart[k];
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(p.counters + b * p.Hkv + h, 1u);
    *sm.flag = (prev == static_cast<unsigned>(p.NS - 1));
  }
  __syncthreads();
  if (*sm.flag) {
    __threadfence();
    combine_global<D>(p, sm, b, h, parts);
    if (tid == 0) p.counters[b * p.Hkv + h] = 0u;
  }
}

template <int D>
size_t smem_bytes(const DecodeParams& p) {
  const size_t stages = static_cast<size_t>(kDecodeWarps) * kDecodeStages * p.stage_bytes;
  // window scores [kMaxGroup][R], or the reserve's scores [kMaxGroup][3W] and
  // member list [3W]
  const size_t win = p.lq_w ? static_cast<size_t>(kMaxGroup + 1) * 3 * p.lq_w * 4
                            : (p.R > 0 ? win_bytes(p.R, D) : 0);
  const size_t merge = static_cast<size_t>(merge_floats<D>()) * 4;   // shares the area
  const size_t weights = static_cast<size_t>(kMaxGroup) * kMaxNS * 4;  // ticket combine
  size_t area = stages > win ? stages : win;
  if (merge > area) area = merge;
  if (weights > area) area = weights;
  return header_bytes(D, rbuf_ctas(p.cluster, p.NS)) + area;
}

// Lets decode_kernel<D, MODE> use up to the device's opt-in shared memory (set
// once per device; never lowered, so any smaller size launches too).
template <int D, int MODE>
cudaError_t allow_smem() {
  static int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_kernel<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           optin);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

template <int D, int MODE>
cudaError_t launch_d(const DecodeParams& p, cudaStream_t s) {
  const size_t bytes = smem_bytes<D>(p);
  if (bytes > 48 * 1024) {
    const cudaError_t e = allow_smem<D, MODE>();
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.NS, p.Hkv, p.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (p.cluster && p.NS > 1) {   // a lone CTA is a cluster of one without the attribute
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = p.NS;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (p.overlap) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, MODE>, p);
}

template <int D, int MODE>
int blocks_per_sm(size_t smem) {
  int n = 0;
  cudaError_t e = allow_smem<D, MODE>();
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, MODE>, kThreads, smem);
  return e == cudaSuccess ? n : -1;
}

template <int D>
int blocks_per_sm_mode(size_t smem, int mode) {
  return mode == kModeLogQuant    ? blocks_per_sm<D, kModeLogQuant>(smem)
         : mode == kModeKeyChannel ? blocks_per_sm<D, kModeKeyChannel>(smem)
                                   : blocks_per_sm<D, kModeTokenWise>(smem);
}

template <int D>
cudaError_t launch_mode(const DecodeParams& p, cudaStream_t s) {
  return p.lq_w  ? launch_d<D, kModeLogQuant>(p, s)
         : p.kpc ? launch_d<D, kModeKeyChannel>(p, s)
                 : launch_d<D, kModeTokenWise>(p, s);
}

}  // namespace

int decode_max_splits() { return kMaxSplits; }
int decode_max_cluster() { return kMaxCluster; }

int decode_blocks_per_sm(int head_dim, size_t smem, int mode) {
  return head_dim == 128 ? blocks_per_sm_mode<128>(smem, mode) : blocks_per_sm_mode<64>(smem, mode);
}

size_t decode_smem_bytes(const DecodeParams& p, int head_dim) {
  return head_dim == 128 ? smem_bytes<128>(p) : smem_bytes<64>(p);
}

cudaError_t launch_decode(const DecodeParams& p, int head_dim, cudaStream_t s) {
  if (head_dim == 128) return launch_mode<128>(p, s);
  if (head_dim == 64) return launch_mode<64>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
