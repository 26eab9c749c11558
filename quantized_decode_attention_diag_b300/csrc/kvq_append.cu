// Quantize-on-append: block-diagonal Walsh-Hadamard rotation of each new K/V
// head vector, token-wise asymmetric INT-b quantization with one fp16 scale and
// zero per (token, head), packed into the paged cache; bf16 recent-token ring.
//
// Method: "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization for Real-World LLM
// Serving" (summary; section 2, rotate before quantizing; section 3, rotation
// and quantization inside the memory pass), RateQuant technical summary,
// Methodology section 3 (separate K and V widths per head), "LogQuant ...",
// Methodology section 2 (full-precision recent window).
//
// Work decomposition: one warp handles 16 vectors that share (KV head, K|V) --
// hence one bit-width -- with two lanes per vector.  Lane u of a pair loads the
// contiguous half [u*D/2, (u+1)*D/2) of the bf16 row (16-byte loads), runs the
// in-register butterflies of the Sylvester transform on it, and a single
// shuffle stage joins the halves when the Hadamard block spans both.  The
// min/max reduction takes one more shuffle; scale and zero are formed with
// explicitly rounded operations (see the header for the exact rule); codes are
// packed in registers and written with 16-byte stores.
#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr float kMagicRound = 12582912.0f;  // 1.5 * 2^23: x + magic rounds x to an integer

template <int D, int NB, int BITS>
__device__ __forceinline__ void append_warp(const AppendParams& p, int h, int kv, int chunk,
                                            int lane) {
  constexpr int E = D / 2;                 // elements per lane
  constexpr int M = (1 << BITS) - 1;
  constexpr int LANE_BYTES = D * BITS / 16;  // packed code bytes per lane
  constexpr int NW = LANE_BYTES / 4;       // 32-bit words per lane
  constexpr int CPW = 32 / BITS;           // codes per word

  const int row = lane >> 1;
  const int u = lane & 1;
  const int r = chunk * 16 + row;
  bool active = r < p.B * p.T;
  int b = 0, t = 0, l0 = 0;
  if (active) {
    b = r / p.T;
    t = r - b * p.T;
    l0 = __ldg(p.seq_lens + b);
    if (l0 < 0 || static_cast<long long>(l0) + p.T > static_cast<long long>(p.max_pages) * kPage) {
      if (u == 0) flag_status(p.status, 0x2);
      active = false;
    }
  }
  const int pos = l0 + t;
  const int len = l0 + p.T;
  const int qlim = p.R ? max(0, len - p.R) : len;

  const uint16_t* in_row =
      (kv ? p.V : p.K) + (static_cast<size_t>(b) * p.T + t) * p.Hkv * D + static_cast<size_t>(h) * D;
  const uint16_t* src = nullptr;
  uint16_t* ring_slot = nullptr;
  int dst = -1;
  if (active) {
    if (pos < qlim) {
      src = in_row;  // never enters the window
      dst = pos;
    } else {
      // enters the ring; the slot's previous occupant (the position of the old
      // window congruent to pos mod R) leaves the window now
      ring_slot = p.window +
                  ((static_cast<size_t>(b) * p.Hkv + h) * 2 + kv) * p.R * D +
                  static_cast<size_t>(pos % p.R) * D;
      const int pold = pos - p.R * ((pos - l0) / p.R + 1);
      if (pold >= 0) {
        src = ring_slot;
        dst = pold;
      }
    }
  }
  uint8_t* seg = nullptr;
  if (dst >= 0) {
    const int pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + dst / kPage);
    if (pid < 0 || pid >= p.num_pages) {
      if (u == 0) flag_status(p.status, 0x1);
      src = nullptr;
      dst = -1;
    } else {
      seg = p.pool + static_cast<size_t>(pid) * p.geom.page_bytes + p.geom.head_off[h];
    }
  }

  // ---- load this lane's half of the row (bf16 -> fp32, exact)
  float v[E];
  if (src != nullptr) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + u * E);
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

  // ---- Sylvester butterflies, natural order: stage hs pairs (i, i + hs)
  constexpr int IN_REG = NB < E ? NB : E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {  // hs = 1
    const float a = v[e], c = v[e + 1];
    v[e] = a + c;
    v[e + 1] = a - c;
  }
#pragma unroll
  for (int hs = 2; hs < IN_REG; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      if (!(e & hs)) addsub2(v[e], v[e + 1], v[e + hs], v[e + hs + 1]);
    }
  }
  if constexpr (NB > E) {  // the block spans both lanes: lane 0 holds the lower half
    const float sgn = u ? -1.f : 1.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(kFullMask, v[e], 1);
      v[e] = __fmaf_rn(sgn, v[e], o);  // u = 0: a + b, u = 1: a - b
    }
  }

  // ---- per-vector min / max over both lanes
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int e = 1; e < E; ++e) {
    mn = fminf(mn, v[e]);
    mx = fmaxf(mx, v[e]);
  }
  mn = fminf(mn, __shfl_xor_sync(kFullMask, mn, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));

  // ---- fp16 zero (round down) and scale (round up)
  const __half zh = __float2half_rd(mn);
  const float zf = __half2float(zh);
  const float span = __fsub_rn(mx, zf);
  const __half sh = __float2half_ru(__fdiv_rn(span, static_cast<float>(M)));
  const float sf = __half2float(sh);
  const float inv = sf > 0.f ? __frcp_rn(sf) : 0.f;

  if (src != nullptr) {
    if (u == 0 && !(isfinite(sf) && isfinite(zf))) flag_status(p.status, 0x4);
    // ---- codes: round-half-even((u - z) * inv) via the magic-number add
    uint32_t words[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      uint32_t acc = 0;
#pragma unroll
      for (int i = 0; i < CPW; ++i) {
        const float f = __fmaf_rn(__fsub_rn(v[w * CPW + i], zf), inv, kMagicRound);
        acc |= (__float_as_uint(f) & static_cast<uint32_t>(M)) << (BITS * i);
      }
      words[w] = acc;
    }
    const int slot = dst % kPage;
    const int kb = D * p.geom.bits[h][0] / 8;  // K code bytes per token
    const int vb = D * p.geom.bits[h][1] / 8;
    uint8_t* cbase = seg + (kv ? kPage * kb : 0) + slot * (D * BITS / 8) + u * LANE_BYTES;
    if constexpr (NW % 4 == 0) {
#pragma unroll
      for (int i = 0; i < NW / 4; ++i)
        reinterpret_cast<uint4*>(cbase)[i] =
            make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
    } else if constexpr (NW == 2) {
      *reinterpret_cast<uint2*>(cbase) = make_uint2(words[0], words[1]);
    } else {
      *reinterpret_cast<uint32_t*>(cbase) = words[0];
    }
    if (u == 0) {
      uint8_t* sz = seg + kPage * (kb + vb) + (kv ? kPage * 4 : 0) + slot * 4;
      *reinterpret_cast<uint32_t*>(sz) = pack_half2(sh, zh);
    }
  }

  // ---- copy the new token into its ring slot (after the old one was read)
  if (ring_slot != nullptr) {
    const uint4* s4 = reinterpret_cast<const uint4*>(in_row + u * E);
    uint4* d4 = reinterpret_cast<uint4*>(ring_slot + u * E);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) d4[i] = s4[i];
  }
}

template <int D, int NB>
__global__ void __launch_bounds__(kAppendWarps * 32)
    append_kernel(const __grid_constant__ AppendParams p) {
  const int warp = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int grp = warp / p.warps_per_group;
  if (grp >= 2 * p.Hkv) return;  // whole warp
  const int chunk = warp - grp * p.warps_per_group;
  const int h = grp >> 1, kv = grp & 1;
  switch (p.geom.bits[h][kv]) {  // warp-uniform
    case 2: append_warp<D, NB, 2>(p, h, kv, chunk, lane); break;
    case 4: append_warp<D, NB, 4>(p, h, kv, chunk, lane); break;
    case 8: append_warp<D, NB, 8>(p, h, kv, chunk, lane); break;
    default: break;
  }
}

template <int D, int NB>
cudaError_t launch(const AppendParams& p, cudaStream_t s) {
  const long long warps = 2ll * p.Hkv * p.warps_per_group;
  const unsigned blocks = static_cast<unsigned>((warps + kAppendWarps - 1) / kAppendWarps);
  append_kernel<D, NB><<<blocks, kAppendWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int head_dim, int had_block, cudaStream_t s) {
  if (head_dim == 128) {
    if (had_block == 128) return launch<128, 128>(p, s);
    if (had_block == 64) return launch<128, 64>(p, s);
    if (had_block == 32) return launch<128, 32>(p, s);
  } else if (head_dim == 64) {
    if (had_block == 64) return launch<64, 64>(p, s);
    if (had_block == 32) return launch<64, 32>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
