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
#include "kvq_quant.cuh"

namespace kvq {

namespace {

template <int D, int NB, int BITS>
__device__ __forceinline__ void append_warp(const AppendParams& p, int h, int kv, int chunk,
                                            int lane) {
  constexpr int E = D / 2;                 // elements per lane
  constexpr int LANE_BYTES = D * BITS / 16;  // packed code bytes per lane
  constexpr int NW = LANE_BYTES / 4;       // 32-bit words per lane

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

  // ---- this lane's half of the row, rotated and quantized with its partner
  float v[E];
  load_half_row<D>(src, u, v);
  uint32_t words[NW];
  __half sh, zh;
  rotate_quantize_half<D, NB, BITS>(v, u, words, sh, zh);

  if (src != nullptr) {
    if (u == 0 && !(isfinite(__half2float(sh)) && isfinite(__half2float(zh))))
      flag_status(p.status, KVQ_DEV_NONFINITE);
    const int slot = dst % kPage;
    const int kb = D * p.geom.bits[h][0] / 8;  // K code bytes per token
    const int vb = D * p.geom.bits[h][1] / 8;
    store_code_words<NW>(seg + (kv ? kPage * kb : 0) + slot * (D * BITS / 8) + u * LANE_BYTES,
                         words);
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
