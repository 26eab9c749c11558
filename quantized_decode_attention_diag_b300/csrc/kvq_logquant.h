// LogQuant log-spaced full-precision selection: which positions of a sequence
// of length n are kept in bf16, and where their rows live in the reserve.
// Shared by the host layer and the kernels.
//
// Method: "LogQuant: Log-Distributed 2-Bit Quantization of KV Cache with
// Superior Accuracy Preservation", Methodology section 2 (a base window W; the
// newest tokens at full precision, older windows selected ever more sparsely;
// a 3W full-precision reserve; when it fills, the older selections are halved)
// and section 4 (A V = A_P V_P: full-precision and quantized tokens combine in
// any order).  Reading: every new token joins the set B; when |B| reaches 3W,
// of the oldest 2W members (by position) every other one is kept, the first of
// each pair.
//
// Closed form for W = 2^a.  The halvings happen at n = 3W, 4W, 5W, ...; after
// k of them (k = 0 for n < 3W, else (n - 3W) / W + 1) the set is
//   B = C_k  U  [(k + 1) W, n)                    (n >= 3W; B = [0, n) before)
// where C_k, W positions, is made of blocks of W positions thinned in place:
//   block 0 = [0, W):     multiples of 2^k (k <= a), else position 0 alone;
//   block b in (k - a, k], b >= 1, at level j = k - b:
//                         b W + 2^(j+1) u,  0 <= u < W / 2^(j+1).
// (Each halving takes the even-indexed half of the oldest 2W members; with W a
// power of two, block b's survivors after j + 1 halvings are every 2^(j+1)-th
// position of the block, and the blocks older than k - a + 1 have been halved
// away except position 0, the first of every pair.)
//
// Reserve rows of one (sequence, KV head, K|V), d bf16 each:
//   rows [0, 3W):          the ring, position p at row p mod 3W -- every
//                          member newer than (k + 1) W, and every member
//                          before the first halving;
//   rows 3W + L W/2 + e:   level buffer L, entry e = (p mod W) / 2: block b
//                          >= 1 in buffer b mod a, block 0 in buffer a.
// A block is copied from the ring into its buffer, its even positions only,
// when the halving that thins it first happens (positions (b + 1) W ... leave
// the ring's reach only W tokens later), and is thinned in place afterwards.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define KVQ_HD __host__ __device__ __forceinline__
#else
#define KVQ_HD inline
#endif

namespace kvq {

// log2 of a power of two w >= 2 (-1 otherwise).
KVQ_HD int lq_log2(int w) {
  if (w < 2 || (w & (w - 1))) return -1;
  int a = 0;
  while ((1 << a) < w) ++a;
  return a;
}

// Halvings done after n appends.
KVQ_HD int lq_halvings(long long n, int w) {
  return n < 3ll * w ? 0 : static_cast<int>((n - 3ll * w) / w) + 1;
}

// Is position p (0 <= p < n) kept at full precision after n appends?
KVQ_HD bool lq_member(long long p, long long n, int w, int a) {
  if (p < 0 || p >= n) return false;
  if (n < 3ll * w) return true;
  const long long k = (n - 3ll * w) / w + 1;
  if (p >= (k + 1) * w) return true;
  const long long blk = p >> a;
  if (blk == 0) return k <= a ? (p & ((1ll << k) - 1)) == 0 : p == 0;
  const long long j = k - blk;
  if (j >= a) return false;
  return ((p & (w - 1)) & ((2ll << j) - 1)) == 0;
}

// lq_member for 32-bit positions and lengths (n < 2^31 - w), as the decode
// kernel's masked rounds use it.
KVQ_HD bool lq_member32(int p, int n, int w, int a) {
  if (p < 0 || p >= n) return false;
  if (n < 3 * w) return true;
  const int k = ((n - 3 * w) >> a) + 1;
  if (p >= ((k + 1) << a)) return true;
  const int blk = p >> a;
  if (blk == 0) return k <= a ? (p & ((1 << k) - 1)) == 0 : p == 0;
  const int j = k - blk;
  if (j >= a) return false;
  return ((p & (w - 1)) & ((2 << j) - 1)) == 0;
}

// Reserve row of member p after n appends (see the header comment).
KVQ_HD int lq_row(long long p, long long n, int w, int a) {
  if (n < 3ll * w) return static_cast<int>(p % (3ll * w));
  const long long k = (n - 3ll * w) / w + 1;
  if (p >= (k + 1) * w) return static_cast<int>(p % (3ll * w));
  const long long blk = p >> a;
  const int level = blk == 0 ? a : static_cast<int>(blk % a);
  return 3 * w + level * (w / 2) + static_cast<int>((p & (w - 1)) >> 1);
}

// lq_row for 32-bit positions and lengths (the decode kernel's member list).
KVQ_HD int lq_row32(int p, int n, int w, int a) {
  if (n < 3 * w) return p % (3 * w);
  const int k = ((n - 3 * w) >> a) + 1;
  if (p >= ((k + 1) << a)) return p % (3 * w);
  const int blk = p >> a;
  const int level = blk == 0 ? a : blk % a;
  return 3 * w + level * (w / 2) + ((p & (w - 1)) >> 1);
}

// The members of B at length n lie in block 0 and from lq_lo() on.
KVQ_HD int lq_lo(long long n, int w, int a) {
  if (n < 3ll * w) return 0;
  const long long k = (n - 3ll * w) / w + 1;
  const long long lo = (k - a + 1) * w;
  return static_cast<int>(lo > w ? lo : w);
}

// Rows of one (sequence, KV head, K|V) plane: the ring and a + 1 level buffers.
KVQ_HD int lq_rows(int w, int a) { return 3 * w + (a + 1) * (w / 2); }

}  // namespace kvq
