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
// Work decomposition: a chunk is 16 vectors that share (KV head, K|V) -- hence
// one bit-width -- quantized by one warp, two lanes per vector.  A wave of
// warps loops over the chunks; each warp prefetches its next chunk's bf16 rows
// into shared memory (cp.async) while it quantizes the current one.  Lane u of
// a pair takes the half [u*D/2, (u+1)*D/2) of its row, runs the in-register
// butterflies of the Sylvester transform on it (packed fp32 pairs), and a
// single shuffle stage joins the halves when the Hadamard block spans both.
// The min/max reduction takes one more shuffle; scale and zero are formed with
// explicitly rounded operations (see the header for the exact rule); codes are
// computed on packed fp32 pairs, packed by shifted sums and written with
// 16-byte stores.
#include <climits>
#include <type_traits>

#include "kvq_logquant.h"
#include "kvq_quant.cuh"

namespace kvq {

namespace {

// This lane's row of chunk c: (KV head, K|V) group and its (sequence, token),
// b = -1 past the batch.  Computed once per chunk.
struct RowRef {
  int grp, b, t;
};
__device__ __forceinline__ RowRef row_ref(const AppendParams& p, int c) {
  const int row = (threadIdx.x & 31) >> 1;
  RowRef rr;
  rr.grp = static_cast<int>(fastdiv(static_cast<uint32_t>(c), p.div_wpg));
  const int r = (c - rr.grp * p.warps_per_group) * 16 + row;
  if (r < p.B * p.T) {
    rr.b = static_cast<int>(fastdiv(static_cast<uint32_t>(r), p.div_T));
    rr.t = r - rr.b * p.T;
  } else {
    rr.b = -1;
    rr.t = 0;
  }
  return rr;
}

// Sequence length before the append (INT_MIN past the batch).
__device__ __forceinline__ int row_len0(const AppendParams& p, const RowRef& rr) {
  return rr.b < 0 ? INT_MIN : __ldg(p.seq_lens + rr.b);
}

// Position the row quantizes (-1: none; see append_chunk).
__device__ __forceinline__ int row_dst(const AppendParams& p, const RowRef& rr, int l0) {
  if (l0 < 0 || l0 > p.cap_tokens - p.T) return -1;   // (INT_MIN: past the batch)
  const int pos = l0 + rr.t, len = l0 + p.T;
  const int qlim = p.R ? max(0, len - p.R) : len;
  if (pos < qlim) return pos;
  return pos - p.R * ((pos - l0) / p.R + 1);   // the ring slot's old occupant, if >= 0
}

// Physical page of that position (-1: none).
__device__ __forceinline__ int row_pid(const AppendParams& p, const RowRef& rr, int l0) {
  const int dst = row_dst(p, rr, l0);
  if (dst < 0) return -1;
  return __ldg(p.page_table + static_cast<size_t>(rr.b) * p.max_pages + dst / kPage);
}

// Row chunk of a warp: 16 vectors (rows) of one (KV head, K|V), 16 consecutive
// (sequence, token) pairs.  The warp's lane pair (row = lane / 2, u = lane % 2)
// quantizes half u of row `row`.  Rows are prefetched into a per-warp
// shared-memory buffer with cp.async, one chunk ahead of the one being
// quantized; 16-byte chunk ci of row r sits at position
// ci ^ ((2 r + ci / (D / 16)) & 7), so that
// the eight lanes of a 16-byte shared-memory phase hit distinct banks.
template <int D>
__device__ __forceinline__ int swz(int row, int ci) {
  return ci ^ ((2 * row + ci / (D / 16)) & 7);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// The chunk's 16 rows are rows r0 .. r0 + 15 of the (sequence, token) order,
// so row k's input is at ((r0 + k) Hkv + h) D.  Each copy instruction moves
// whole rows: D / 8 lanes per 16-byte chunk of a row, 32 / (D / 8) rows at a
// time, every 32-byte sector read once.
template <int D>
__device__ __forceinline__ void prefetch_chunk(const AppendParams& p, int c, uint4* buf) {
  constexpr int LPR = D / 8;                   // lanes per row
  constexpr int RPI = 32 / LPR;                // rows per instruction
  const int lane = threadIdx.x & 31;
  // chunk c: group grp, rows blk * 16 ..
  const int grp = static_cast<int>(fastdiv(static_cast<uint32_t>(c), p.div_wpg));
  const int blk = c - grp * p.warps_per_group;
  const int h = grp >> 1, kv = grp & 1;
  const int rows = p.B * p.T;                  // <= 2^28 (checked on the host)
  const int ci = lane % LPR, k0 = lane / LPR;
  const int rl = blk * 16 + k0;                // this lane's first row
  // piece ci of row r is at (r Hkv + h) D elements + ci pieces; the rows a lane
  // copies are RPI apart, RPI Hkv D elements
  const uint4* src = reinterpret_cast<const uint4*>((kv ? p.V : p.K) +
                                                    (static_cast<size_t>(rl) * p.Hkv + h) * D) + ci;
  const size_t step = static_cast<size_t>(RPI) * p.Hkv * (D / 8);
#pragma unroll
  for (int i = 0; i < 16 / RPI; ++i) {
    const int k = RPI * i + k0;
    if (rl + RPI * i < rows) cp_async16(buf + k * (D / 8) + swz<D>(k, ci), src + i * step);
  }
}

// load_row_top from the staged row (both halves; see kvq_quant.cuh)
template <int D>
__device__ __forceinline__ void row_top_from_smem(const uint4* buf, int row, int u,
                                                  float (&v)[D / 2]) {
  const float sgn = u ? -1.f : 1.f;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    const uint4 lo = buf[row * (D / 8) + swz<D>(row, i)];
    const uint4 hi = buf[row * (D / 8) + swz<D>(row, D / 16 + i)];
    top_stage8(lo, hi, sgn, v + 8 * i);
  }
}

template <int D>
__device__ __forceinline__ void half_row_from_smem(const uint4* buf, int row, int u,
                                                   float (&v)[D / 2]) {
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    const uint4 w = buf[row * (D / 8) + swz<D>(row, u * (D / 16) + i)];
    v[8 * i + 0] = bf16lo(w.x); v[8 * i + 1] = bf16hi(w.x);
    v[8 * i + 2] = bf16lo(w.y); v[8 * i + 3] = bf16hi(w.y);
    v[8 * i + 4] = bf16lo(w.z); v[8 * i + 5] = bf16hi(w.z);
    v[8 * i + 6] = bf16lo(w.w); v[8 * i + 7] = bf16hi(w.w);
  }
}

// Quantize-on-append of chunk c whose input rows are in `buf`.
template <int D, int NB, int BITS>
__device__ __forceinline__ void append_chunk(const AppendParams& p, const RowRef& rr,
                                             const uint4* buf, int l0, int pid) {
  constexpr int E = D / 2;                 // elements per lane
  constexpr int LANE_BYTES = D * BITS / 16;  // packed code bytes per lane
  constexpr int NW = LANE_BYTES / 4;       // 32-bit words per lane
  const int lane = threadIdx.x & 31, row = lane >> 1, u = lane & 1;
  const int h = rr.grp >> 1, kv = rr.grp & 1;
  const int b = rr.b < 0 ? 0 : rr.b, t = rr.t;
  bool active = rr.b >= 0;
  if (active &&
      (l0 < 0 || l0 > p.cap_tokens - p.T)) {
    if (u == 0) flag_status(p.status, KVQ_DEV_BAD_LENGTH);
    active = false;
  }
  if (!active) l0 = 0;
  const int pos = l0 + t;
  const int len = l0 + p.T;
  const int qlim = p.R ? max(0, len - p.R) : len;

  // where the quantized vector comes from (the input row in smem, or the ring
  // slot it leaves) and which position it fills; ring slot the input enters
  const uint16_t* from_ring = nullptr;
  uint16_t* ring_slot = nullptr;
  int dst = -1;
  if (active) {
    if (pos < qlim) {
      // never enters the window: quantized straight from the input row
      dst = pos;
    } else {
      // enters the ring; the slot's previous occupant (the position of the old
      // window congruent to pos mod R) leaves the window now
      ring_slot = p.window + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + kv) * p.R * D +
                  static_cast<size_t>(pos % p.R) * D;
      const int pold = pos - p.R * ((pos - l0) / p.R + 1);
      if (pold >= 0) {
        from_ring = ring_slot;
        dst = pold;
      }
    }
  }
  // LogQuant mode (R = 0 here, every token quantized): a member of B after the
  // append keeps its bf16 row in the reserve (`window`)
  uint16_t* lq_dst = nullptr;
  if (active && p.lq_w && lq_member(pos, len, p.lq_w, p.lq_a)) {
    lq_dst = p.window + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + kv) * p.lq_rows * D +
             static_cast<size_t>(lq_row(pos, len, p.lq_w, p.lq_a)) * D;
  }
  uint8_t* seg = nullptr;
  if (dst >= 0) {
    if (pid < 0 || pid >= p.num_pages) {
      if (u == 0) flag_status(p.status, KVQ_DEV_BAD_PAGE);
      from_ring = nullptr;
      dst = -1;
    } else {
      // a page is under 1 MB: one 32 x 32 -> 64-bit multiply-add
      seg = p.pool + static_cast<uint32_t>(pid) * static_cast<size_t>(
                         static_cast<uint32_t>(p.geom.page_bytes)) + p.geom.head_off[h];
    }
  }

  // ---- this lane's half of the row, rotated and quantized with its partner;
  //      rows past the batch quantize whatever the buffer holds, unused
  float v[E];
  if constexpr (NB > E) {                // the block is the whole vector: top stage first
    if (from_ring == nullptr) {
      row_top_from_smem<D>(buf, row, u, v);
    } else {
      load_row_top<D>(from_ring, u, v);  // only with a window
    }
  } else {
    if (from_ring == nullptr) {
      half_row_from_smem<D>(buf, row, u, v);
    } else {
      load_half_row<D>(from_ring, u, v); // only with a window
    }
  }
  uint32_t words[NW];
  __half sh, zh;
  rotate_quantize_half<D, NB, BITS>(v, u, words, sh, zh);

  if (dst >= 0) {
    const int slot = dst % kPage;
    const int kb = D * p.geom.bits[h][0] / 8;  // K code bytes per token
    const int vb = D * p.geom.bits[h][1] / 8;
    store_code_words<NW>(seg + (kv ? kPage * kb : 0) + slot * (D * BITS / 8) + u * LANE_BYTES,
                         words);
    uint32_t* sz = reinterpret_cast<uint32_t*>(seg + kPage * (kb + vb) + (kv ? kPage * 4 : 0) +
                                               slot * 4);
    const uint32_t szv = pack_half2(sh, zh);
    if (u == 0) *sz = szv;
    if (!(isfinite(__half2float(sh)) && isfinite(__half2float(zh))) && u == 0)
      flag_status(p.status, KVQ_DEV_NONFINITE);
  }

  // ---- copy the new token into its ring slot (after the old one was read),
  //      or into its LogQuant reserve row
  uint16_t* row_dst = ring_slot != nullptr ? ring_slot : lq_dst;
  if (row_dst != nullptr) {
    uint4* d4 = reinterpret_cast<uint4*>(row_dst) + u * (D / 16);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) d4[i] = buf[row * (D / 8) + swz<D>(row, u * (D / 16) + i)];
  }
}

template <int D, int NB>
__global__ void __launch_bounds__(kAppendWarps * 32, kAppendCtas)
    append_kernel(const __grid_constant__ AppendParams p) {
  // [warps][kAppendBufs][16 rows][D / 8] 16-byte chunks: the chunk being
  // quantized and the next kAppendBufs - 1 in flight
  extern __shared__ uint4 abuf[];
  const int warp = threadIdx.x >> 5;
  const int total = 2 * p.Hkv * p.warps_per_group;
  const int stride = gridDim.x * kAppendWarps;
  uint4* mine = abuf + warp * kAppendBufs * 16 * (D / 8);
  auto slot = [&](int i) { return mine + (i % kAppendBufs) * 16 * (D / 8); };
  int c = blockIdx.x * kAppendWarps + warp;
  // metadata pipeline: lengths two chunks ahead, page ids one chunk ahead
  RowRef rc = row_ref(p, c < total ? c : 0);
  RowRef rn = row_ref(p, c + stride < total ? c + stride : 0);
  int l0_c = c < total ? row_len0(p, rc) : INT_MIN;
  int l0_n = c + stride < total ? row_len0(p, rn) : INT_MIN;
  int pid_c = c < total ? row_pid(p, rc, l0_c) : -1;
  // rows of the first kAppendBufs - 1 chunks
  for (int i = 0; i < kAppendBufs - 1; ++i) {
    const int ci = c + i * stride;
    if (ci < total) prefetch_chunk<D>(p, ci, slot(i));
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int it = 0; c < total; c += stride, ++it) {
    const int cn = c + stride, cnn = cn + stride;
    const RowRef rnn = row_ref(p, cnn < total ? cnn : 0);
    int pid_n = -1, l0_nn = INT_MIN;
    if (cn < total) pid_n = row_pid(p, rn, l0_n);
    if (cnn < total) l0_nn = row_len0(p, rnn);
    const int cf = c + (kAppendBufs - 1) * stride;   // the chunk whose rows go out now
    if (cf < total) prefetch_chunk<D>(p, cf, slot(it + kAppendBufs - 1));
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(kAppendBufs - 1) : "memory");
    __syncwarp();
    const uint4* buf = slot(it);
    switch (p.geom.bits[rc.grp >> 1][rc.grp & 1]) {  // warp-uniform
      case 2: append_chunk<D, NB, 2>(p, rc, buf, l0_c, pid_c); break;
      case 4: append_chunk<D, NB, 4>(p, rc, buf, l0_c, pid_c); break;
      case 8: append_chunk<D, NB, 8>(p, rc, buf, l0_c, pid_c); break;
      default: break;
    }
    __syncwarp();
    rc = rn;
    rn = rnn;
    l0_c = l0_n;
    pid_c = pid_n;
    l0_n = l0_nn;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// LogQuant carry, one CTA per (sequence, KV head): the halvings this append
// performs (k0 .. k1 - 1, from the lengths before and after) each thin a block
// for the first time; that block's even positions still in the reserve's ring
// -- those older than this append -- move to the block's level buffer (the
// append itself writes the rows of its own tokens where they end up).  Blocks
// halved away again before the end are skipped; the first halving also moves
// block 0.  Copying a few positions the later halvings drop is harmless.
template <int D>
__global__ void __launch_bounds__(128) lq_carry_kernel(const __grid_constant__ AppendParams p) {
  const int b = blockIdx.x, h = blockIdx.y;
  const int l0 = __ldg(p.seq_lens + b);
  if (l0 < 0 || static_cast<long long>(l0) + p.T > static_cast<long long>(p.max_pages) * kPage)
    return;                                    // the append reports the bad length
  const int w = p.lq_w, a = p.lq_a, half = w / 2;
  const long long n = static_cast<long long>(l0) + p.T;
  const int k0 = lq_halvings(l0, w), k1 = lq_halvings(n, w);
  if (k1 == k0) return;
  constexpr int C = D / 8;                     // uint4 chunks per row
  for (int kv = 0; kv < 2; ++kv) {
    uint16_t* plane = p.window + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + kv) * p.lq_rows * D;
    for (int i = max(k0, k1 - a); i < k1; ++i) {
      const int blk = 1 + i;                   // alive at the end: blk > k1 - a
      for (int pass = 0; pass < (i == 0 ? 2 : 1); ++pass) {
        const int bb = pass ? 0 : blk;         // the first halving moves block 0 too
        const int level = bb == 0 ? a : bb % a;
        for (int idx = threadIdx.x; idx < half * C; idx += blockDim.x) {
          const int v = idx / C, ci = idx - v * C;
          const long long q = static_cast<long long>(bb) * w + 2 * v;
          if (q >= l0) continue;               // a token of this append
          const uint4* src = reinterpret_cast<const uint4*>(plane + (q % (3ll * w)) * D) + ci;
          uint4* dst = reinterpret_cast<uint4*>(plane + (3 * w + level * half + v) * D) + ci;
          *dst = *src;
        }
      }
    }
  }
}

// ---------------------------------------------------- key-per-channel mode
// RateQuant technical summary, Methodology section 3 (KIVI: symmetric
// per-channel keys, asymmetric per-token values); "LogQuant ...", section 5
// (key-per-channel).  A page is quantized once all its 16 positions have left
// the window: the quantized prefix of length L is Q(L) = 16 floor(max(L - R,
// 0) / 16), and positions Q(L) .. L - 1 keep bf16 rows in a ring of R + 16 rows
// (p.R here), slot p mod (R + 16).
__device__ __forceinline__ int kpc_prefix(int len, int ring) {
  return kPage * (max(0, len - (ring - kPage)) / kPage);
}

// Sequence length before the append (p.lens_after: seq_lens already count the
// appended tokens, as in a decode step).
__device__ __forceinline__ int append_len0(const AppendParams& p, int b) {
  return __ldg(p.seq_lens + b) - (p.lens_after ? p.T : 0);
}

// The bf16 row of position pos of (b, h, kv): the ring (older than the
// append) or the appended input.
template <int D>
__device__ __forceinline__ const uint16_t* kpc_row(const AppendParams& p, int b, int h, int kv,
                                                   int pos, int l0) {
  if (pos < l0)
    return p.window + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + kv) * p.R * D +
           static_cast<size_t>(pos % p.R) * D;
  return (kv ? p.V : p.K) + ((static_cast<size_t>(b) * p.T + (pos - l0)) * p.Hkv + h) * D;
}

// One CTA per (page completed by this append, KV head, sequence); warp 0
// quantizes the page's 16 keys per channel, warp 1 its 16 values token-wise.
// Lanes 2 r and 2 r + 1 hold halves of token r (the append's layout).  Keys:
// the rotated halves go to shared memory, lane j forms the scale of channels
// j, j + 32, ... (max |u| over the 16 tokens / (2^(b-1) - 1), fp16 rounded up)
// and its fp32 reciprocal, then every lane codes its own half.
template <int D, int NB>
__global__ void __launch_bounds__(64) kpc_page_kernel(const __grid_constant__ AppendParams p) {
  constexpr int E = D / 2;
  constexpr int LD = D + 4;                    // padded row of the key buffer (floats)
  __shared__ __align__(16) float kbuf[kPage * LD];
  __shared__ float invs[D];
  const int b = blockIdx.z, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = lane >> 1, u = lane & 1;
  const int l0 = append_len0(p, b), len = l0 + p.T;
  if (l0 < 0 || static_cast<long long>(len) > static_cast<long long>(p.max_pages) * kPage) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(p.status, KVQ_DEV_BAD_LENGTH);
    return;
  }
  const int pg = kpc_prefix(l0, p.R) / kPage + static_cast<int>(blockIdx.x);
  if (pg >= kpc_prefix(len, p.R) / kPage) return;
  const int pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
  if (pid < 0 || pid >= p.num_pages) {
    if (threadIdx.x == 0) flag_status(p.status, KVQ_DEV_BAD_PAGE);
    return;
  }
  const int bk = p.geom.bits[h][0], bv = p.geom.bits[h][1];
  const int kb = D * bk / 8, vb = D * bv / 8;
  uint8_t* seg = p.pool + static_cast<size_t>(pid) * p.geom.page_bytes + p.geom.head_off[h];
  const int kv = warp;
  const uint16_t* src = kpc_row<D>(p, b, h, kv, pg * kPage + r, l0);
  float v[E];
  if constexpr (NB > E) load_row_top<D>(src, u, v);
  else load_half_row<D>(src, u, v);

  if (kv == 1) {                               // values: the token-wise rule
    uint8_t* vsz = seg + kPage * (kb + vb) + 2 * D + r * 4;
    auto quant = [&](auto bits_tag) {
      constexpr int BITS = decltype(bits_tag)::value;
      constexpr int NW = D * BITS / 64;
      uint32_t words[NW];
      __half sh, zh;
      rotate_quantize_half<D, NB, BITS>(v, u, words, sh, zh);
      store_code_words<NW>(seg + kPage * kb + r * (D * BITS / 8) + u * (D * BITS / 16), words);
      if (u == 0) {
        *reinterpret_cast<uint32_t*>(vsz) = pack_half2(sh, zh);
        if (!(isfinite(__half2float(sh)) && isfinite(__half2float(zh))))
          flag_status(p.status, KVQ_DEV_NONFINITE);
      }
    };
    if (bv == 2) quant(std::integral_constant<int, 2>{});
    else if (bv == 4) quant(std::integral_constant<int, 4>{});
    else quant(std::integral_constant<int, 8>{});
    return;
  }

  // keys: per-channel scales over the page's 16 tokens
  rotate_half<D, NB>(v);
#pragma unroll
  for (int i = 0; i < E / 4; ++i)
    *reinterpret_cast<float4*>(kbuf + r * LD + u * E + 4 * i) =
        make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  __syncwarp();
  const float qmax = static_cast<float>((1 << (bk - 1)) - 1);
  __half* scales = reinterpret_cast<__half*>(seg + kPage * (kb + vb));
  bool bad = false;
#pragma unroll
  for (int m = 0; m < D / 32; ++m) {
    const int ch = lane + 32 * m;
    float amax = 0.f;
#pragma unroll
    for (int t = 0; t < kPage; ++t) amax = fmaxf(amax, fabsf(kbuf[t * LD + ch]));
    const __half sh = __float2half_ru(__fdiv_rn(amax, qmax));
    const float sf = __half2float(sh);
    bad |= !isfinite(sf);
    scales[ch] = sh;
    invs[ch] = sf > 0.f ? __frcp_rn(sf) : 0.f;
  }
  if (bad) flag_status(p.status, KVQ_DEV_NONFINITE);
  __syncwarp();
  auto codes = [&](auto bits_tag) {
    constexpr int BITS = decltype(bits_tag)::value;
    constexpr int NW = D * BITS / 64;
    uint32_t words[NW];
    quantize_channels_half<D, BITS>(v, invs + u * E, words);
    store_code_words<NW>(seg + r * (D * BITS / 8) + u * (D * BITS / 16), words);
  };
  if (bk == 2) codes(std::integral_constant<int, 2>{});
  else if (bk == 4) codes(std::integral_constant<int, 4>{});
  else codes(std::integral_constant<int, 8>{});
}

// After kpc_page_kernel: the appended positions that stay in bf16 (from
// max(l0, Q(len)) on) into the ring.  Grid (rows / 4, Hkv, B), one warp per
// position copying its K and V rows.
template <int D>
__global__ void __launch_bounds__(128) kpc_ring_kernel(const __grid_constant__ AppendParams p) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int l0 = append_len0(p, b), len = l0 + p.T;
  if (l0 < 0 || static_cast<long long>(len) > static_cast<long long>(p.max_pages) * kPage) return;
  const int pos = max(l0, kpc_prefix(len, p.R)) + static_cast<int>(blockIdx.x) * 4 + warp;
  if (pos >= len) return;
  constexpr int C = D / 8;                     // 16-byte chunks per row
  for (int idx = lane; idx < 2 * C; idx += 32) {
    const int kv = idx / C, ci = idx - kv * C;
    const uint4* from = reinterpret_cast<const uint4*>(
        (kv ? p.V : p.K) + ((static_cast<size_t>(b) * p.T + (pos - l0)) * p.Hkv + h) * D);
    uint4* to = reinterpret_cast<uint4*>(p.window + ((static_cast<size_t>(b) * p.Hkv + h) * 2 + kv) *
                                                        p.R * D +
                                         static_cast<size_t>(pos % p.R) * D);
    to[ci] = from[ci];
  }
}

template <int D, int NB>
cudaError_t launch_kpc(const AppendParams& p, cudaStream_t s) {
  // pages a sequence can complete: (T + 15) / 16 + 1; rows it can keep: R + 15
  const int pages = (p.T + kPage - 1) / kPage + 1;
  kpc_page_kernel<D, NB><<<dim3(pages, p.Hkv, p.B), 64, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = min(p.T, p.R - 1);
  kpc_ring_kernel<D><<<dim3((rows + 3) / 4, p.Hkv, p.B), 128, 0, s>>>(p);
  return cudaGetLastError();
}

int sm_count_cached() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int D, int NB>
cudaError_t launch(const AppendParams& p, cudaStream_t s) {
  constexpr size_t smem = static_cast<size_t>(kAppendWarps) * kAppendBufs * 16 * D * 2;
  static int attr_set[64] = {0};   // per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(append_kernel<D, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = 1;
  }
  const long long chunks = 2ll * p.Hkv * p.warps_per_group;
  // one resident wave of warps (kAppendCtas CTAs per SM), each looping over its chunks
  const long long wave = static_cast<long long>(kAppendCtas) * kAppendWarps * sm_count_cached();
  const long long warps = chunks < wave ? chunks : wave;
  const unsigned blocks = static_cast<unsigned>((warps + kAppendWarps - 1) / kAppendWarps);
  append_kernel<D, NB><<<blocks, kAppendWarps * 32, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lq_carry(const AppendParams& p, int head_dim, cudaStream_t s) {
  const dim3 grid(p.B, p.Hkv);
  if (head_dim == 128) lq_carry_kernel<128><<<grid, 128, 0, s>>>(p);
  else if (head_dim == 64) lq_carry_kernel<64><<<grid, 128, 0, s>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_kpc_append(const AppendParams& p, int head_dim, int had_block, cudaStream_t s) {
  if (head_dim == 128) {
    if (had_block == 128) return launch_kpc<128, 128>(p, s);
    if (had_block == 64) return launch_kpc<128, 64>(p, s);
    if (had_block == 32) return launch_kpc<128, 32>(p, s);
    if (had_block == 1) return launch_kpc<128, 1>(p, s);
  } else if (head_dim == 64) {
    if (had_block == 64) return launch_kpc<64, 64>(p, s);
    if (had_block == 32) return launch_kpc<64, 32>(p, s);
    if (had_block == 1) return launch_kpc<64, 1>(p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_append(const AppendParams& p, int head_dim, int had_block, cudaStream_t s) {
  if (head_dim == 128) {
    if (had_block == 128) return launch<128, 128>(p, s);
    if (had_block == 64) return launch<128, 64>(p, s);
    if (had_block == 32) return launch<128, 32>(p, s);
    if (had_block == 1) return launch<128, 1>(p, s);
  } else if (head_dim == 64) {
    if (had_block == 64) return launch<64, 64>(p, s);
    if (had_block == 32) return launch<64, 32>(p, s);
    if (had_block == 1) return launch<64, 1>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
