// Rotation and quantization of one K or V head vector by a pair of lanes,
// shared by the append kernel and the decode step (sm_103a).
//
// Method: "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization for Real-World LLM
// Serving" (section 2: rotate each head vector with a block-diagonal Hadamard
// transform before quantizing it token-wise) and the RateQuant technical
// summary, Methodology section 3 (asymmetric per-token quantization with its
// own bit-width per head and K/V).  The exact rule (Sylvester order,
// unnormalised transform, fp16 zero rounded down and scale rounded up, codes
// by round-half-even of (u - z) * (1 / s) in fp32) is stated in kvq.h.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

constexpr float kMagicRound = 12582912.0f;  // 1.5 * 2^23: x + magic rounds x to an integer

// The top stage on 8 bf16 pairs: v_k = lo_k + hi_k (sgn = 1) or lo_k - hi_k.
__device__ __forceinline__ void top_stage8(const uint4& lo, const uint4& hi, float sgn, float* v) {
  const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w}, b[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __fmaf_rn(sgn, bf16lo(b[j]), bf16lo(a[j]));
    v[2 * j + 1] = __fmaf_rn(sgn, bf16hi(b[j]), bf16hi(a[j]));
  }
}

// Lane u (0 or 1) of a pair loads half u of a bf16 head vector (dims
// [u D/2, (u+1) D/2)) as exact fp32; zeros when row is null.
template <int D>
__device__ __forceinline__ void load_half_row(const uint16_t* row, int u, float (&v)[D / 2]) {
  constexpr int E = D / 2;
  if (row != nullptr) {
    const uint4* s4 = reinterpret_cast<const uint4*>(row + u * E);
    uint4 w[D / 16];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) w[i] = s4[i];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      v[8 * i + 0] = bf16lo(w[i].x); v[8 * i + 1] = bf16hi(w[i].x);
      v[8 * i + 2] = bf16lo(w[i].y); v[8 * i + 3] = bf16hi(w[i].y);
      v[8 * i + 4] = bf16lo(w[i].z); v[8 * i + 5] = bf16hi(w[i].z);
      v[8 * i + 6] = bf16lo(w[i].w); v[8 * i + 7] = bf16hi(w[i].w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = 0.f;
  }
}

// Lane u of a pair loads dims [u D/2, (u+1) D/2) of the top Sylvester stage of
// a bf16 head vector x whose Hadamard block is the whole vector: x_i + x_{i+D/2}
// (u = 0) or x_i - x_{i+D/2} (u = 1), each rounded once to fp32.  The stages
// of the transform commute, so this one comes first.  Both halves are read,
// and no value crosses lanes.
template <int D>
__device__ __forceinline__ void load_row_top(const uint16_t* row, int u, float (&v)[D / 2]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(row);
  const float sgn = u ? -1.f : 1.f;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    const uint4 lo = s4[i], hi = s4[D / 16 + i];
    top_stage8(lo, hi, sgn, v + 8 * i);
  }
}

// The Sylvester butterflies of the stages inside a lane's half (natural
// order: stage hs pairs (i, i + hs); NB == 1: no rotation, u = x).  When the
// block spans both halves (NB > D / 2) the caller has applied the top stage
// already (load_row_top).
// Blocks no wider than a quarter row (2 <= NB <= D / 4) put elements j and
// j + D / 4 of a lane's half in different blocks that take the same stages, so
// every stage runs on the packed pairs (v[j], v[j + D/4]); each element still
// sees the same additions in the same order.
template <int D, int NB>
constexpr bool kCrossPairs = NB >= 2 && NB <= D / 4;

template <int D, int NB>
__device__ __forceinline__ void rotate_half(float (&v)[D / 2]) {
  constexpr int E = D / 2;                 // elements per lane
  constexpr int IN_REG = NB < E ? NB : E;
  if constexpr (kCrossPairs<D, NB>) {
#pragma unroll
    for (int hs = 1; hs < NB; hs <<= 1) {
#pragma unroll
      for (int j = 0; j < E / 2; ++j)
        if (!(j & hs)) addsub2(v[j], v[j + E / 2], v[j + hs], v[j + hs + E / 2]);
    }
    return;
  }
  if constexpr (NB >= 2) {
#pragma unroll
    for (int e = 0; e < E; e += 2) {  // hs = 1
      const float a = v[e], c = v[e + 1];
      v[e] = a + c;
      v[e + 1] = a - c;
    }
  }
#pragma unroll
  for (int hs = 2; hs < IN_REG; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      if (!(e & hs)) addsub2(v[e], v[e + 1], v[e + hs], v[e + hs + 1]);
    }
  }
}

// Rotates the vector held by the lane pair (lane ^ 1 is the partner; every
// lane of the warp must call this) and quantizes it: this lane's packed codes
// (half u of the row, D * BITS / 16 bytes as 32-bit words), and the pair's
// fp16 scale and zero.  When the block spans both halves (NB > D / 2) the
// caller has applied the top stage already (load_row_top); the other stages
// then stay inside the lane.
template <int D, int NB, int BITS>
__device__ __forceinline__ void rotate_quantize_half(float (&v)[D / 2], int u,
                                                     uint32_t (&words)[D * BITS / 64], __half& sh,
                                                     __half& zh) {
  constexpr int E = D / 2;                 // elements per lane
  constexpr int M = (1 << BITS) - 1;
  constexpr int NW = D * BITS / 64;        // 32-bit words per lane
  constexpr int CPW = 32 / BITS;           // codes per word

  rotate_half<D, NB>(v);

  // ---- per-vector min / max over both lanes (eight independent chains of
  //      three-input min / max: min and max are exact, so the order does not
  //      matter)
  constexpr int RK = E >= 8 ? 8 : E;
  float mnk[RK], mxk[RK];
#pragma unroll
  for (int j = 0; j < RK; ++j) mnk[j] = mxk[j] = v[j];
  int e0 = RK;
#pragma unroll
  for (; e0 + 2 * RK <= E; e0 += 2 * RK) {
#pragma unroll
    for (int j = 0; j < RK; ++j) {
      mnk[j] = fmin3(mnk[j], v[e0 + j], v[e0 + RK + j]);
      mxk[j] = fmax3(mxk[j], v[e0 + j], v[e0 + RK + j]);
    }
  }
#pragma unroll
  for (; e0 < E; e0 += RK) {
#pragma unroll
    for (int j = 0; j < RK; ++j) {
      mnk[j] = fminf(mnk[j], v[e0 + j]);
      mxk[j] = fmaxf(mxk[j], v[e0 + j]);
    }
  }
  float mn = mnk[0], mx = mxk[0];
#pragma unroll
  for (int j = 1; j + 1 < RK; j += 2) {
    mn = fmin3(mn, mnk[j], mnk[j + 1]);
    mx = fmax3(mx, mxk[j], mxk[j + 1]);
  }
  if constexpr (RK % 2 == 0) {
    mn = fminf(mn, mnk[RK - 1]);
    mx = fmaxf(mx, mxk[RK - 1]);
  }
  mn = fminf(mn, __shfl_xor_sync(kFullMask, mn, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));

  // ---- fp16 zero (round down) and scale (round up)
  zh = __float2half_rd(mn);
  const float zf = __half2float(zh);
  const float span = __fsub_rn(mx, zf);
  sh = __float2half_ru(__fdiv_rn(span, static_cast<float>(M)));
  const float sf = __half2float(sh);
  const float inv = sf > 0.f ? __frcp_rn(sf) : 0.f;

  // ---- codes: round-half-even((u - z) * inv) via the magic-number add; the
  //      result's bits are 0x4B400000 + code, so the packed word is the sum of
  //      the bit patterns shifted into place minus the shifted constants.
  //      There is no clamp: z rounded down and s rounded up keep (u - z) * inv
  //      within [0, M + 1/2), so every code lies in [0, M] (a CPU test drives
  //      the same fp32 rule through extreme spans, subnormal scales included)
  constexpr uint32_t kMagicBits = 0x4B400000u;
  uint32_t ksum = 0;
#pragma unroll
  for (int i = 0; i < CPW; ++i) ksum += kMagicBits << (BITS * i);
  if constexpr (kCrossPairs<D, NB>) {
    // the rotation's pairs (v[j], v[j + E/2]): codes j and j + E/2 sit at the
    // same place of words E/2 / CPW apart
    static_assert((E / 2) % CPW == 0, "half of a lane's elements fill whole words");
#pragma unroll
    for (int w = 0; w < NW; ++w) words[w] = 0u - ksum;
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      uint32_t f0, f1;
      subfma2(v[j], v[j + E / 2], zf, inv, kMagicRound, f0, f1);
      words[j / CPW] += f0 << (BITS * (j % CPW));
      words[(j + E / 2) / CPW] += f1 << (BITS * (j % CPW));
    }
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      uint32_t acc = 0u - ksum;
#pragma unroll
      for (int i = 0; i < CPW; i += 2) {
        uint32_t f0, f1;
        subfma2(v[w * CPW + i], v[w * CPW + i + 1], zf, inv, kMagicRound, f0, f1);
        acc += (f0 << (BITS * i)) + (f1 << (BITS * (i + 1)));
      }
      words[w] = acc;
    }
  }
  (void)M;
}

// Key-per-channel mode: this lane's packed codes of its E = D / 2 rotated
// values for the page's channel reciprocals inv[] (dims [u E, u E + E)): code
// round-half-even(v * inv) stored as c + 2^(BITS-1), by the magic-number add
// (the offset is even, so ties still go to the even code).  The scale rounded
// up keeps |v * inv| <= 2^(BITS-1) - 1 + 2^-20, so no clamp is needed.
template <int D, int BITS>
__device__ __forceinline__ void quantize_channels_half(const float (&v)[D / 2], const float* inv,
                                                       uint32_t (&words)[D * BITS / 64]) {
  constexpr int NW = D * BITS / 64;
  constexpr int CPW = 32 / BITS;
  constexpr float kMagicOff = kMagicRound + float(1 << (BITS - 1));
  constexpr uint32_t kMagicBits = 0x4B400000u;
  uint32_t ksum = 0;
#pragma unroll
  for (int i = 0; i < CPW; ++i) ksum += kMagicBits << (BITS * i);
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    uint32_t acc = 0u - ksum;
#pragma unroll
    for (int i = 0; i < CPW; ++i) {
      const float f = __fmaf_rn(v[w * CPW + i], inv[w * CPW + i], kMagicOff);
      acc += __float_as_uint(f) << (BITS * i);
    }
    words[w] = acc;
  }
}

// Stores this lane's packed code words (NW of them) at dst (16-, 8- or
// 4-byte aligned according to their size).
template <int NW>
__device__ __forceinline__ void store_code_words(uint8_t* dst, const uint32_t (&words)[NW]) {
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i)
      reinterpret_cast<uint4*>(dst)[i] =
          make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
  } else if constexpr (NW == 2) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = words[0];
  }
}

// ------------------------------------------------------------------------
// The same rotation and quantization for two vectors at once, one per
// half-warp (lanes 0-15: vector A with BITS_A, lanes 16-31: vector B with
// BITS_B); lane l of a half holds the 8 (D = 128) or 4 (D = 64) consecutive
// elements [F (l % 16), F (l % 16) + F).  Every element goes through the same
// fp32 operations as in rotate_quantize_half (a + b and a - b stage by stage,
// the same min / max, scale, zero and rounding), so the codes are identical;
// only the placement across lanes differs.  Writes this lane's codes (F codes,
// little-endian, packed into `code_bits` bits of `codes`) and the vector's
// (s, z).  Every lane of the warp must call it; nb is the Hadamard block.
template <int D>
__device__ __forceinline__ void rotate_quantize_halfwarp(float (&v)[D / 16], int nb, int bits,
                                                         uint32_t (&codes)[2], __half& sh,
                                                         __half& zh) {
  constexpr int F = D / 16;   // elements per lane
  const int lane = threadIdx.x & 31;
  // a block of the whole vector takes its top stage (hs = D / 2, lanes l and
  // l ^ 8) first, the order of the pair routine's load_row_top
  constexpr int kTopM = D / 2 / F;
  const bool top_first = nb == D;
  if (top_first) {
    const float sgn = (lane & kTopM) ? -1.f : 1.f;
#pragma unroll
    for (int e = 0; e < F; ++e) {
      const float o = __shfl_xor_sync(kFullMask, v[e], kTopM);
      v[e] = __fmaf_rn(sgn, v[e], o);   // lower: a + b, upper: a - b
    }
  }
  // butterflies inside the lane: stages hs < F
#pragma unroll
  for (int hs = 1; hs < F; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < F; ++e) {
      if (!(e & hs) && hs < nb) {
        const float a = v[e], c = v[e + hs];
        v[e] = a + c;
        v[e + hs] = a - c;
      }
    }
  }
  // across lanes: stage hs = F m pairs lanes l and l ^ m (within the half)
  for (int m = 1; m * F < nb; m <<= 1) {
    if (top_first && m == kTopM) break;   // done first
    const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int e = 0; e < F; ++e) {
      const float o = __shfl_xor_sync(kFullMask, v[e], m);
      v[e] = __fmaf_rn(sgn, v[e], o);   // lower: a + b, upper: a - b
    }
  }
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int e = 1; e < F; ++e) {
    mn = fminf(mn, v[e]);
    mx = fmaxf(mx, v[e]);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(kFullMask, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, o));
  }
  const float M = static_cast<float>((1 << bits) - 1);
  zh = __float2half_rd(mn);
  const float zf = __half2float(zh);
  const float span = __fsub_rn(mx, zf);
  sh = __float2half_ru(__fdiv_rn(span, M));
  const float sf = __half2float(sh);
  const float inv = sf > 0.f ? __frcp_rn(sf) : 0.f;
  const uint32_t mask = (1u << bits) - 1u;
  uint64_t acc = 0;
#pragma unroll
  for (int e = 0; e < F; ++e) {
    const float f = __fmaf_rn(__fsub_rn(v[e], zf), inv, kMagicRound);
    acc |= static_cast<uint64_t>(__float_as_uint(f) & mask) << (bits * e);
  }
  codes[0] = static_cast<uint32_t>(acc);
  codes[1] = static_cast<uint32_t>(acc >> 32);
}

}  // namespace kvq
