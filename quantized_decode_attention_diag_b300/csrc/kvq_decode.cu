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
// covers the bf16 window.  Each CTA writes an online-softmax partial
// (m, l, acc[d]) per query head; the last CTA of (b, h) to finish (an atomic
// ticket, no waiting) merges them and writes o.
//
// Quantized split, per warp: pages w, w + 4, ... of the split stream through a
// 4-stage ring of shared-memory buffers, each filled by one cp.async.bulk of
// the (page, head) segment (TMA engine, completion on an mbarrier).  A page is
// 16 tokens = the M dimension of one m16n8k16 tensor-core MMA:
//   scores:  S[16 tok x 8] = C_K[16 tok x d] * Qhl[d x 8]
//   output:  O[d x 8]     += C_V^T[d x 16 tok] * Phl[16 tok x 8]
// where the 8 columns are the 4 query heads of the GQA group, each split into
// an fp16 "hi" part and an fp16 "lo" remainder (x = hi + lo to ~22 bits), so
// the group fills the n8 tile exactly and the fp32 accumulators keep fp32
// accuracy.  Codes enter the MMA as exact fp16 integers; the scale and zero are
// folded outside the MMA: score = s (q'' . c) + z sum(q''),
// sum_t p_t deq(v_t) = sum_t (p_t s_t) c_t + sum_t p_t z_t.
#include <math_constants.h>

#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kThreads = kDecodeWarps * 32;
constexpr int kMaxSplits = 256;

struct Smem {
  float* qtab;        // [kMaxGroup][D]   rotated, scaled queries (or raw for the window)
  float* qsum;        // [kMaxGroup]
  int* flag;
  uint64_t* bars;     // [warps][stages]
  uint8_t* area;      // stage buffers / merge / window / combine scratch
};

template <int D>
__device__ __forceinline__ Smem carve(uint8_t* base, int stage_bytes) {
  Smem s;
  s.qtab = reinterpret_cast<float*>(base);
  s.qsum = s.qtab + kMaxGroup * D;
  s.flag = reinterpret_cast<int*>(s.qsum + kMaxGroup);
  s.bars = reinterpret_cast<uint64_t*>(base + kMaxGroup * D * 4 + 64);
  s.area = base + kMaxGroup * D * 4 + 64 + kDecodeWarps * kDecodeStages * 8;
  s.area = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s.area) + 127) & ~uintptr_t(127));
  (void)stage_bytes;
  return s;
}

__host__ __device__ constexpr int header_bytes(int d) {
  return ((d * kMaxGroup * 4 + 64 + kDecodeWarps * kDecodeStages * 8) + 127) / 128 * 128 + 128;
}

// ------------------------------------------------------------ load helpers --
template <int NBYTES>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t* w) {
  if constexpr (NBYTES % 16 == 0) {
#pragma unroll
    for (int i = 0; i < NBYTES / 16; ++i) {
      const uint4 x = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
    }
  } else if constexpr (NBYTES == 8) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    w[0] = x.x; w[1] = x.y;
  } else if constexpr (NBYTES == 4) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else {
    static_assert(NBYTES == 2, "unsupported row slice");
    w[0] = *reinterpret_cast<const uint16_t*>(p);
  }
}

// ------------------------------------------------- K codes -> fp16 pairs ----
// Pairs come out in the order whose dims kpair_dims() reports.
template <int BITS, int NWORDS>
__device__ __forceinline__ void kconv(const uint32_t* w, uint32_t* pr) {
#pragma unroll
  for (int i = 0; i < NWORDS; ++i) {
    const uint32_t x = w[i];
    if constexpr (BITS == 4) {
      const uint32_t y = x >> 8;
      pr[4 * i + 0] = h2_sub1024(lop_or_magic(x, 0x000f000fu));
      pr[4 * i + 1] = h2_unscale<4>(lop_or_magic(x, 0x00f000f0u));
      pr[4 * i + 2] = h2_sub1024(lop_or_magic(y, 0x000f000fu));
      pr[4 * i + 3] = h2_unscale<4>(lop_or_magic(y, 0x00f000f0u));
    } else if constexpr (BITS == 2) {
      const uint32_t y = x >> 8;
      pr[8 * i + 0] = h2_sub1024(lop_or_magic(x, 0x00030003u));
      pr[8 * i + 1] = h2_unscale<2>(lop_or_magic(x, 0x000c000cu));
      pr[8 * i + 2] = h2_unscale<4>(lop_or_magic(x, 0x00300030u));
      pr[8 * i + 3] = h2_unscale<6>(lop_or_magic(x, 0x00c000c0u));
      pr[8 * i + 4] = h2_sub1024(lop_or_magic(y, 0x00030003u));
      pr[8 * i + 5] = h2_unscale<2>(lop_or_magic(y, 0x000c000cu));
      pr[8 * i + 6] = h2_unscale<4>(lop_or_magic(y, 0x00300030u));
      pr[8 * i + 7] = h2_unscale<6>(lop_or_magic(y, 0x00c000c0u));
    } else {
      pr[2 * i + 0] = h2_sub1024(__byte_perm(x, 0x64646464u, 0x4140));
      pr[2 * i + 1] = h2_sub1024(__byte_perm(x, 0x64646464u, 0x4342));
    }
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
// Pair i = dim i of the thread's slice, (token 1 in the low half, token 2 high).
template <int BITS, int NWORDS>
__device__ __forceinline__ void vconv(const uint32_t* w1, const uint32_t* w2, uint32_t* pr) {
#pragma unroll
  for (int i = 0; i < NWORDS; ++i) {
    const uint32_t x1 = w1[i], x2 = w2[i];
    if constexpr (BITS == 4) {
      const uint32_t a = __byte_perm(x1, x2, 0x5410), a8 = a >> 8;
      const uint32_t b = __byte_perm(x1, x2, 0x7632), b8 = b >> 8;
      pr[8 * i + 0] = h2_sub1024(lop_or_magic(a, 0x000f000fu));
      pr[8 * i + 1] = h2_unscale<4>(lop_or_magic(a, 0x00f000f0u));
      pr[8 * i + 2] = h2_sub1024(lop_or_magic(a8, 0x000f000fu));
      pr[8 * i + 3] = h2_unscale<4>(lop_or_magic(a8, 0x00f000f0u));
      pr[8 * i + 4] = h2_sub1024(lop_or_magic(b, 0x000f000fu));
      pr[8 * i + 5] = h2_unscale<4>(lop_or_magic(b, 0x00f000f0u));
      pr[8 * i + 6] = h2_sub1024(lop_or_magic(b8, 0x000f000fu));
      pr[8 * i + 7] = h2_unscale<4>(lop_or_magic(b8, 0x00f000f0u));
    } else if constexpr (BITS == 2) {
      // a word holds 16 dims; the 2-byte slice (head_dim 64) holds 8
      const uint32_t a = __byte_perm(x1, x2, 0x5410), a8 = a >> 8;
      pr[16 * i + 0] = h2_sub1024(lop_or_magic(a, 0x00030003u));
      pr[16 * i + 1] = h2_unscale<2>(lop_or_magic(a, 0x000c000cu));
      pr[16 * i + 2] = h2_unscale<4>(lop_or_magic(a, 0x00300030u));
      pr[16 * i + 3] = h2_unscale<6>(lop_or_magic(a, 0x00c000c0u));
      pr[16 * i + 4] = h2_sub1024(lop_or_magic(a8, 0x00030003u));
      pr[16 * i + 5] = h2_unscale<2>(lop_or_magic(a8, 0x000c000cu));
      pr[16 * i + 6] = h2_unscale<4>(lop_or_magic(a8, 0x00300030u));
      pr[16 * i + 7] = h2_unscale<6>(lop_or_magic(a8, 0x00c000c0u));
      const uint32_t b = __byte_perm(x1, x2, 0x7632), b8 = b >> 8;
      pr[16 * i + 8] = h2_sub1024(lop_or_magic(b, 0x00030003u));
      pr[16 * i + 9] = h2_unscale<2>(lop_or_magic(b, 0x000c000cu));
      pr[16 * i + 10] = h2_unscale<4>(lop_or_magic(b, 0x00300030u));
      pr[16 * i + 11] = h2_unscale<6>(lop_or_magic(b, 0x00c000c0u));
      pr[16 * i + 12] = h2_sub1024(lop_or_magic(b8, 0x00030003u));
      pr[16 * i + 13] = h2_unscale<2>(lop_or_magic(b8, 0x000c000cu));
      pr[16 * i + 14] = h2_unscale<4>(lop_or_magic(b8, 0x00300030u));
      pr[16 * i + 15] = h2_unscale<6>(lop_or_magic(b8, 0x00c000c0u));
    } else {
      pr[4 * i + 0] = h2_sub1024(lop_or_magic(__byte_perm(x1, x2, 0x4400), 0x00ff00ffu));
      pr[4 * i + 1] = h2_sub1024(lop_or_magic(__byte_perm(x1, x2, 0x5511), 0x00ff00ffu));
      pr[4 * i + 2] = h2_sub1024(lop_or_magic(__byte_perm(x1, x2, 0x6622), 0x00ff00ffu));
      pr[4 * i + 3] = h2_sub1024(lop_or_magic(__byte_perm(x1, x2, 0x7733), 0x00ff00ffu));
    }
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
// qtab <- the group's queries scaled by softmax_scale * log2(e) (and, for the
// quantized splits, rotated: q'' = H q / n); qsum[i] = sum_d qtab[i][d].
template <int D>
__device__ void query_prologue(const DecodeParams& p, const Smem& sm, bool rotate) {
  const int tid = threadIdx.x;
  if (rotate) {
    const int nb = p.had_block;
    for (int hs = 1; hs < nb; hs <<= 1) {
      for (int idx = tid; idx < kMaxGroup * (D / 2); idx += kThreads) {
        const int i = idx / (D / 2), r = idx - i * (D / 2);
        const int lo = (r / hs) * 2 * hs + (r % hs);
        const float a = sm.qtab[i * D + lo], c = sm.qtab[i * D + lo + hs];
        sm.qtab[i * D + lo] = a + c;
        sm.qtab[i * D + lo + hs] = a - c;
      }
      __syncthreads();
    }
  }
  const float qscale = rotate ? p.scale_log2 / static_cast<float>(p.had_block) : p.scale_log2;
  for (int idx = tid; idx < kMaxGroup * D; idx += kThreads) sm.qtab[idx] *= qscale;
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  float s = 0.f;
  for (int d = lane; d < D; d += 32) s += sm.qtab[warp * D + d];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFullMask, s, o);
  if (lane == 0) sm.qsum[warp] = s;
  __syncthreads();
}

// 2^x with the hardware approximation (relative error ~2^-22); 2^-inf = 0
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ quantized split
template <int D, int BK, int BV>
__device__ void quant_split(const DecodeParams& p, const Smem& sm, int b, int h, int split,
                            int lq, float* part) {
  constexpr int KB = D * BK / 8;                 // K code bytes per token
  constexpr int VB = D * BV / 8;
  constexpr int CHUNK = kPage * (KB + VB + 8);   // one (page, head) segment
  constexpr int NJ = D / 16;                     // MMAs along d
  constexpr int KSLICE = KB / 4;                 // bytes of a token row per k-slot group
  constexpr int VSLICE = VB / 8;                 // bytes of a token row per dim group
  constexpr int KWORDS = KSLICE >= 4 ? KSLICE / 4 : 1;
  constexpr int VWORDS = VSLICE >= 4 ? VSLICE / 4 : 1;
  // pairs vconv produces (>= 2 * NJ; only head_dim 64 with 2-bit values makes
  // more than are used, from the zero upper half of a 2-byte slice)
  constexpr int VPAIRS = (BV == 2 ? 16 : BV == 4 ? 8 : 4) * VWORDS;
  static_assert(VPAIRS >= 2 * NJ, "value slice too small");
  constexpr int NST = kDecodeStages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;

  // ---- this warp's pages: first + 4 k, k < nk; their ids in registers,
  //      32 per chunk (lane i holds page k = 32 * chunk + i)
  const int npages = (lq + kPage - 1) / kPage;
  const int pg0 = split * p.pages_per_split;
  const int pg1 = min(npages, pg0 + p.pages_per_split);
  const int first = pg0 + warp;
  const int nk = pg1 > first ? (pg1 - first + kDecodeWarps - 1) / kDecodeWarps : 0;
  const int32_t* ptab = p.page_table + static_cast<size_t>(b) * p.max_pages + first;
  auto load_chunk = [&](int ch) -> int {
    const int kk = 32 * ch + lane;
    return kk < nk ? __ldg(ptab + kDecodeWarps * kk) : -1;
  };
  int chunk = 0;
  int pid_cur = load_chunk(0);
  int pid_nxt = nk > 32 ? load_chunk(1) : -1;
  auto pid_of = [&](int kk) -> int {  // warp-uniform kk in [32 chunk, 32 chunk + 64)
    const int v = (kk >> 5) == chunk ? pid_cur : pid_nxt;
    return __shfl_sync(kFullMask, v, kk & 31);
  };
  uint8_t* stages = sm.area + static_cast<size_t>(warp) * NST * p.stage_bytes;
  uint64_t* bars = sm.bars + warp * NST;
  const uint8_t* head_base = p.pool + p.geom.head_off[h];
  auto issue = [&](int kk, int pid) {  // lane 0 only
    uint64_t* bar = bars + (kk % NST);
    if (pid < 0 || pid >= p.num_pages) {
      flag_status(p.status, 0x1);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
      return;
    }
    mbar_expect_tx(bar, CHUNK);
    bulk_g2s(stages + (kk % NST) * p.stage_bytes,
             head_base + static_cast<size_t>(pid) * p.geom.page_bytes, CHUNK, bar);
  };
  // start streaming before the query prologue
  for (int kk = 0; kk < nk && kk < NST; ++kk) {
    const int pid = pid_of(kk);
    if (lane == 0) issue(kk, pid);
  }

  query_prologue<D>(p, sm, true);

  // ---- B fragments of the rotated, scaled query (hi / lo split), column n = g
  uint32_t bq[NJ][2];
  {
    const float* qh = sm.qtab + (g >> 1) * D;
    const bool lo_part = g & 1;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        int d0, d1;
        kpair_dims<D, BK>(c, 2 * j + s2, d0, d1);
        float x0 = qh[d0], x1 = qh[d1];
        if (lo_part) { x0 -= hi_part(x0); x1 -= hi_part(x1); }
        const __half2 hv = __floats2half2_rn(x0, x1);
        bq[j][s2] = *reinterpret_cast<const uint32_t*>(&hv);
      }
    }
  }
  const float qs = sm.qsum[c];

  float m = -CUDART_INF_F, l = 0.f, zacc = 0.f;
  float oacc[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

  // scores of tokens (g, g + 8) of one staged page, log2 units, -inf if masked
  auto scores = [&](const uint8_t* st, int tok0, float& sc0, float& sc1) {
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t w0[KWORDS], w1[KWORDS];
    lds_words<KSLICE>(st + g * KB + c * KSLICE, w0);
    lds_words<KSLICE>(st + (g + 8) * KB + c * KSLICE, w1);
    uint32_t p0[2 * NJ], p1[2 * NJ];
    kconv<BK, KWORDS>(w0, p0);
    kconv<BK, KWORDS>(w1, p1);
#pragma unroll
    for (int j = 0; j < NJ; j += 2) {   // two independent accumulator chains
      const uint32_t x[4] = {p0[2 * j], p1[2 * j], p0[2 * j + 1], p1[2 * j + 1]};
      mma_16816(a0, x, bq[j][0], bq[j][1]);
      const uint32_t y[4] = {p0[2 * j + 2], p1[2 * j + 2], p0[2 * j + 3], p1[2 * j + 3]};
      mma_16816(a1, y, bq[j + 1][0], bq[j + 1][1]);
    }
    const uint32_t* ksz = reinterpret_cast<const uint32_t*>(st + kPage * (KB + VB));
    const float2 k0 = __half22float2(*reinterpret_cast<const __half2*>(ksz + g));
    const float2 k1 = __half22float2(*reinterpret_cast<const __half2*>(ksz + g + 8));
    sc0 = tok0 + g < lq ? __fmaf_rn(k0.x, (a0[0] + a0[1]) + (a1[0] + a1[1]), k0.y * qs)
                        : -CUDART_INF_F;
    sc1 = tok0 + g + 8 < lq ? __fmaf_rn(k1.x, (a0[2] + a0[3]) + (a1[2] + a1[3]), k1.y * qs)
                            : -CUDART_INF_F;
  };
  // p (already exp'ed, 0 if masked) -> B fragments of the PV MMA; l, zacc
  auto pfrag = [&](const uint8_t* st, float p0, float p1, uint32_t& pb0, uint32_t& pb1) {
    const uint32_t* vsz = reinterpret_cast<const uint32_t*>(st + kPage * (KB + VB)) + kPage;
    const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(vsz + g));
    const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(vsz + g + 8));
    const float ps0 = p0 > 0.f ? p0 * v0.x : 0.f;   // masked tokens: garbage s, z ignored
    const float ps1 = p1 > 0.f ? p1 * v1.x : 0.f;
    if (p0 > 0.f) zacc = __fmaf_rn(p0, v0.y, zacc);
    if (p1 > 0.f) zacc = __fmaf_rn(p1, v1.y, zacc);
    l += p0 + p1;
    const __half2 hi = __floats2half2_rn(ps0, ps1);
    const float2 hf = __half22float2(hi);
    const __half2 lo = __floats2half2_rn(ps0 - hf.x, ps1 - hf.y);
    const uint32_t hip = *reinterpret_cast<const uint32_t*>(&hi);
    const uint32_t lop = *reinterpret_cast<const uint32_t*>(&lo);
    const int src1 = 4 * c + (g >> 1), src2 = src1 + 16;
    const uint32_t h1 = __shfl_sync(kFullMask, hip, src1);
    const uint32_t l1 = __shfl_sync(kFullMask, lop, src1);
    const uint32_t h2 = __shfl_sync(kFullMask, hip, src2);
    const uint32_t l2 = __shfl_sync(kFullMask, lop, src2);
    pb0 = (g & 1) ? l1 : h1;
    pb1 = (g & 1) ? l2 : h2;
  };
  // values: tokens (c, c+8) and (c+4, c+12), dims [g D/8, (g+1) D/8)
  auto pv = [&](const uint8_t* st, uint32_t pb0, uint32_t pb1) {
    const uint8_t* vc = st + kPage * KB;
    uint32_t a0[VWORDS], a1[VWORDS], b0[VWORDS], b1[VWORDS];
    lds_words<VSLICE>(vc + c * VB + g * VSLICE, a0);
    lds_words<VSLICE>(vc + (c + 8) * VB + g * VSLICE, a1);
    lds_words<VSLICE>(vc + (c + 4) * VB + g * VSLICE, b0);
    lds_words<VSLICE>(vc + (c + 12) * VB + g * VSLICE, b1);
    uint32_t pa[VPAIRS], pb[VPAIRS];
    vconv<BV, VWORDS>(a0, a1, pa);
    vconv<BV, VWORDS>(b0, b1, pb);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const uint32_t x[4] = {pa[2 * j], pa[2 * j + 1], pb[2 * j], pb[2 * j + 1]};
      mma_16816(oacc[j], x, pb0, pb1);
    }
  };

  bool timed_out = false;
  int k = 0;
  for (; k < nk; k += 2) {                    // two pages per iteration
    if (k >= 32 * (chunk + 1)) {
      ++chunk;
      pid_cur = pid_nxt;
      pid_nxt = load_chunk(chunk + 1);
    }
    const bool has_b = k + 1 < nk;            // warp-uniform
    const int pid_a = pid_of(k);
    const int pid_b = has_b ? pid_of(k + 1) : -1;
    bool ok = mbar_wait_bounded(bars + (k % NST), (k / NST) & 1);
    if (has_b) ok = mbar_wait_bounded(bars + ((k + 1) % NST), ((k + 1) / NST) & 1) && ok;
    if (!__all_sync(kFullMask, ok)) {
      timed_out = true;
      break;
    }
    const bool va = pid_a >= 0 && pid_a < p.num_pages;
    const bool vb = has_b && pid_b >= 0 && pid_b < p.num_pages;
    const uint8_t* sta = stages + (k % NST) * p.stage_bytes;
    const uint8_t* stb = stages + ((k + 1) % NST) * p.stage_bytes;
    const int tok_a = (first + kDecodeWarps * k) * kPage;
    const int tok_b = tok_a + kDecodeWarps * kPage;

    float sa0 = -CUDART_INF_F, sa1 = -CUDART_INF_F, sb0 = -CUDART_INF_F, sb1 = -CUDART_INF_F;
    if (va) scores(sta, tok_a, sa0, sa1);
    if (vb) scores(stb, tok_b, sb0, sb1);

    // online softmax over the 32 tokens, per query head c
    const float mnew = fmaxf(m, warp_max_group(fmaxf(fmaxf(sa0, sa1), fmaxf(sb0, sb1))));
    const bool grow = mnew > m;
    if (__any_sync(kFullMask, grow)) {
      const float alpha = grow ? ex2(m - mnew) : 1.f;
      l *= alpha;
      zacc *= alpha;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        oacc[j][0] *= alpha; oacc[j][1] *= alpha; oacc[j][2] *= alpha; oacc[j][3] *= alpha;
      }
      m = mnew;
    }
    if (va) {
      uint32_t pb0, pb1;
      pfrag(sta, sa0 > -CUDART_INF_F ? ex2(sa0 - m) : 0.f,
            sa1 > -CUDART_INF_F ? ex2(sa1 - m) : 0.f, pb0, pb1);
      pv(sta, pb0, pb1);
    }
    if (vb) {
      uint32_t pb0, pb1;
      pfrag(stb, sb0 > -CUDART_INF_F ? ex2(sb0 - m) : 0.f,
            sb1 > -CUDART_INF_F ? ex2(sb1 - m) : 0.f, pb0, pb1);
      pv(stb, pb0, pb1);
    }
    __syncwarp();
    if (k + NST < nk) {
      const int pid = pid_of(k + NST);
      if (lane == 0) issue(k + NST, pid);
    }
    if (k + 1 + NST < nk) {
      const int pid = pid_of(k + 1 + NST);
      if (lane == 0) issue(k + 1 + NST, pid);
    }
  }
  if (timed_out) {
    if (lane == 0) flag_status(p.status, 0x8);
    for (int kk = k; kk < nk && kk < k + NST; ++kk)
      (void)mbar_wait_bounded(bars + (kk % NST), (kk / NST) & 1);
  }

  // ---- warp partial -> shared, then CTA merge -> global partial
  l = warp_sum_group(l);
  zacc = warp_sum_group(zacc);
  __syncthreads();  // every warp is done with its stage buffers
  float* mrg = reinterpret_cast<float*>(sm.area);   // [warps][kMaxGroup][D + 2]
  float* wrow = mrg + (warp * kMaxGroup + c) * (D + 2);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    wrow[g * (D / 8) + 2 * j] = oacc[j][0] + oacc[j][1] + zacc;
    wrow[g * (D / 8) + 2 * j + 1] = oacc[j][2] + oacc[j][3] + zacc;
  }
  if (g == 0) {
    wrow[D] = m;
    wrow[D + 1] = l;
  }
  __syncthreads();
  for (int idx = tid; idx < p.G * (D + 2); idx += kThreads) {
    const int i = idx / (D + 2), d = idx - i * (D + 2);
    float mm = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) mm = fmaxf(mm, mrg[(w * kMaxGroup + i) * (D + 2) + D]);
    float r = 0.f;
    if (d == D) {
      r = mm;
    } else if (mm != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float* row = mrg + (w * kMaxGroup + i) * (D + 2);
        const float mw = row[D];
        if (mw != -CUDART_INF_F) r = __fmaf_rn(ex2(mw - mm), row[d], r);
      }
    }
    part[i * (D + 2) + d] = r;
  }
}

// ------------------------------------------------------------- window split
template <int D>
__device__ void window_split(const DecodeParams& p, const Smem& sm, int b, int h, int len, int lq,
                             float* part) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nw = len - lq;
  float* sc = reinterpret_cast<float*>(sm.area);   // [kMaxGroup][R]
  const int R = p.R;
  const uint16_t* kring = p.window + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + 0) * R * D;
  const uint16_t* vring = kring + static_cast<size_t>(R) * D;
  for (int t = tid; t < nw; t += kThreads) {
    const uint4* kr = reinterpret_cast<const uint4*>(kring + static_cast<size_t>((lq + t) % R) * D);
    float acc[kMaxGroup] = {0.f, 0.f, 0.f, 0.f};
    for (int i8 = 0; i8 < D / 8; ++i8) {
      const uint4 w = kr[i8];
      const float x[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                          bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
      for (int i = 0; i < kMaxGroup; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i] = __fmaf_rn(sm.qtab[i * D + 8 * i8 + e], x[e], acc[i]);
    }
#pragma unroll
    for (int i = 0; i < kMaxGroup; ++i) sc[i * R + t] = acc[i];
  }
  __syncthreads();
  if (warp < p.G) {  // warp i: softmax statistics of query head i
    float mm = -CUDART_INF_F;
    for (int t = lane; t < nw; t += 32) mm = fmaxf(mm, sc[warp * R + t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFullMask, mm, o));
    float ll = 0.f;
    for (int t = lane; t < nw; t += 32) {
      const float e = exp2f(sc[warp * R + t] - mm);
      sc[warp * R + t] = e;
      ll += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ll += __shfl_xor_sync(kFullMask, ll, o);
    if (lane == 0) {
      part[warp * (D + 2) + D] = nw > 0 ? mm : -CUDART_INF_F;
      part[warp * (D + 2) + D + 1] = ll;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < p.G * D; idx += kThreads) {
    const int i = idx / D, d = idx - i * D;
    float acc = 0.f;
    for (int t = 0; t < nw; ++t) {
      const uint16_t raw = vring[static_cast<size_t>((lq + t) % R) * D + d];
      acc = __fmaf_rn(sc[i * R + t], __uint_as_float(static_cast<uint32_t>(raw) << 16), acc);
    }
    part[i * (D + 2) + d] = acc;
  }
}

// -------------------------------------------------------------- the combine
template <int D>
__device__ void combine(const DecodeParams& p, const Smem& sm, int b, int h,
                        const float* parts) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* wts = reinterpret_cast<float*>(sm.area);         // [kMaxGroup][NS]
  float* lsum = wts + kMaxGroup * (kMaxSplits + 1);       // [kMaxGroup]
  float* orot = lsum + kMaxGroup;                          // [kMaxGroup][D]
  const int NS = p.NS;
  if (warp < p.G) {
    float mm = -CUDART_INF_F;
    for (int s = lane; s < NS; s += 32)
      mm = fmaxf(mm, __ldcg(parts + (static_cast<size_t>(s) * kMaxGroup + warp) * (D + 2) + D));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFullMask, mm, o));
    float ll = 0.f;
    for (int s = lane; s < NS; s += 32) {
      const float* row = parts + (static_cast<size_t>(s) * kMaxGroup + warp) * (D + 2);
      const float ms = __ldcg(row + D);
      const float w = (ms == -CUDART_INF_F) ? 0.f : exp2f(ms - mm);
      wts[warp * (kMaxSplits + 1) + s] = w;
      if (w != 0.f) ll = __fmaf_rn(w, __ldcg(row + D + 1), ll);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ll += __shfl_xor_sync(kFullMask, ll, o);
    if (lane == 0) lsum[warp] = ll;
  }
  __syncthreads();
  for (int idx = tid; idx < p.G * D; idx += kThreads) {
    const int i = idx / D, d = idx - i * D;
    float acc = 0.f;
    for (int s = 0; s < p.S; ++s) {
      const float w = wts[i * (kMaxSplits + 1) + s];
      if (w != 0.f)
        acc = __fmaf_rn(w, __ldcg(parts + (static_cast<size_t>(s) * kMaxGroup + i) * (D + 2) + d),
                        acc);
    }
    orot[i * D + d] = acc;
  }
  __syncthreads();
  // undo the rotation of the value accumulator: x = H u / n (block-diagonal)
  const int nb = p.had_block;
  for (int hs = 1; hs < nb; hs <<= 1) {
    for (int idx = tid; idx < p.G * (D / 2); idx += kThreads) {
      const int i = idx / (D / 2), r = idx - i * (D / 2);
      const int lo = (r / hs) * 2 * hs + (r % hs);
      const float a = orot[i * D + lo], c = orot[i * D + lo + hs];
      orot[i * D + lo] = a + c;
      orot[i * D + lo + hs] = a - c;
    }
    __syncthreads();
  }
  const float inv_nb = 1.f / static_cast<float>(nb);
  for (int idx = tid; idx < p.G * D; idx += kThreads) {
    const int i = idx / D, d = idx - i * D;
    float val = orot[i * D + d] * inv_nb;
    if (p.R > 0) {
      const float ww = wts[i * (kMaxSplits + 1) + p.S];
      if (ww != 0.f)
        val = __fmaf_rn(ww, __ldcg(parts + (static_cast<size_t>(p.S) * kMaxGroup + i) * (D + 2) + d),
                        val);
    }
    const float ll = lsum[i];
    p.o[(static_cast<size_t>(b) * p.Hq + h * p.G + i) * D + d] = ll > 0.f ? val / ll : 0.f;
  }
}

// -------------------------------------------------------------- the kernel --
template <int D>
__global__ void __launch_bounds__(kThreads, 4) decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const Smem sm = carve<D>(smem_raw, p.stage_bytes);
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;

  int len = __ldg(p.seq_lens + b);
  if (len < 0 || len > p.max_pages * kPage) {
    if (tid == 0) flag_status(p.status, 0x2);
    len = 0;
  }
  const int lq = p.R ? max(0, len - p.R) : len;
  float* parts = p.partials + (static_cast<size_t>(b) * p.Hkv + h) * p.NS * kMaxGroup * (D + 2);
  float* part = parts + static_cast<size_t>(split) * kMaxGroup * (D + 2);
  const bool is_window = split >= p.S;

  // queries of the group (rotated and scaled inside the splits' prologue)
  for (int idx = tid; idx < kMaxGroup * D; idx += kThreads) {
    const int i = idx / D, d = idx - i * D;
    float x = 0.f;
    if (i < p.G) {
      const size_t off = (static_cast<size_t>(b) * p.Hq + h * p.G + i) * D + d;
      x = p.q_fp32 ? reinterpret_cast<const float*>(p.q)[off]
                   : __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p.q)[off]) << 16);
    }
    sm.qtab[idx] = x;
  }
  if (tid == 0) {
    for (int i = 0; i < kDecodeWarps * kDecodeStages; ++i) mbar_init(sm.bars + i, 1);
    mbar_init_fence();
  }
  __syncthreads();

  if (is_window) {
    query_prologue<D>(p, sm, false);
    window_split<D>(p, sm, b, h, len, lq, part);
  } else {
    const int bk = p.geom.bits[h][0], bv = p.geom.bits[h][1];
    switch (bk * 16 + bv) {
      case 0x22: quant_split<D, 2, 2>(p, sm, b, h, split, lq, part); break;
      case 0x24: quant_split<D, 2, 4>(p, sm, b, h, split, lq, part); break;
      case 0x28: quant_split<D, 2, 8>(p, sm, b, h, split, lq, part); break;
      case 0x42: quant_split<D, 4, 2>(p, sm, b, h, split, lq, part); break;
      case 0x44: quant_split<D, 4, 4>(p, sm, b, h, split, lq, part); break;
      case 0x48: quant_split<D, 4, 8>(p, sm, b, h, split, lq, part); break;
      case 0x82: quant_split<D, 8, 2>(p, sm, b, h, split, lq, part); break;
      case 0x84: quant_split<D, 8, 4>(p, sm, b, h, split, lq, part); break;
      case 0x88: quant_split<D, 8, 8>(p, sm, b, h, split, lq, part); break;
      default: break;
    }
  }

  // ---- ticket: the last CTA of (b, h) merges every split
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(p.counters + b * p.Hkv + h, 1u);
    *sm.flag = (prev == static_cast<unsigned>(p.NS - 1));
  }
  __syncthreads();
  if (*sm.flag) {
    __threadfence();
    combine<D>(p, sm, b, h, parts);
    if (tid == 0) p.counters[b * p.Hkv + h] = 0u;
  }
}

template <int D>
size_t smem_bytes(const DecodeParams& p) {
  const size_t stages = static_cast<size_t>(kDecodeWarps) * kDecodeStages * p.stage_bytes;
  const size_t merge = static_cast<size_t>(kDecodeWarps) * kMaxGroup * (D + 2) * 4;
  const size_t win = static_cast<size_t>(kMaxGroup) * p.R * 4;
  const size_t comb = (static_cast<size_t>(kMaxGroup) * (kMaxSplits + 1) + kMaxGroup +
                       kMaxGroup * D) * 4;
  size_t area = stages;
  if (merge > area) area = merge;
  if (win > area) area = win;
  if (comb > area) area = comb;
  return header_bytes(D) + area;
}

// Lets decode_kernel<D> use up to the device's opt-in shared memory (set once
// per device; never lowered, so any smaller size launches too).
template <int D>
cudaError_t allow_smem() {
  static int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, cudaStream_t s) {
  const size_t bytes = smem_bytes<D>(p);
  if (bytes > 48 * 1024) {
    const cudaError_t e = allow_smem<D>();
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(p.NS, p.Hkv, p.B);
  decode_kernel<D><<<grid, kThreads, bytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

int decode_max_splits() { return kMaxSplits; }

int decode_blocks_per_sm(int head_dim, size_t smem) {
  int n = 0;
  cudaError_t e;
  if (head_dim == 128) {
    e = allow_smem<128>();
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<128>, kThreads, smem);
  } else {
    e = allow_smem<64>();
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<64>, kThreads, smem);
  }
  return e == cudaSuccess ? n : -1;
}

size_t decode_smem_bytes(const DecodeParams& p, int head_dim) {
  return head_dim == 128 ? smem_bytes<128>(p) : smem_bytes<64>(p);
}

cudaError_t launch_decode(const DecodeParams& p, int head_dim, cudaStream_t s) {
  if (head_dim == 128) return launch_d<128>(p, s);
  if (head_dim == 64) return launch_d<64>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
