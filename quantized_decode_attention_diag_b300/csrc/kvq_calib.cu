// Distortion calibration: kvq_distortion() (sm_103a).
//
// Method: RateQuant technical summary, Methodology section 3 (fit the distortion
// model D(b) = alpha * beta^-b of the quantizer actually used, per K and V
// component, on a small calibration set) and section 4 (5 bit-widths).  The
// quantizer measured is the cache's ("SAW-INT4: System-Aware 4-Bit KV-Cache
// Quantization for Real-World LLM Serving", section 2: block-diagonal Hadamard
// rotation, then token-wise asymmetric quantization): unnormalised Sylvester
// rotation u of each bf16 vector, z = fp16 round-down(min u), s = fp16
// round-up((max u - z) / M), c = round-half-even((u - z) * (1 / s)) with the
// difference and the reciprocal rounded to fp32, deq = c s + z.
//
// One half-warp per vector (16 lanes, D / 16 elements each); CTA (g, h) takes
// the vectors t = g, g + G, ... of KV head h and accumulates, per width, the
// squared error of every vector; the CTA's sums go to the output with one fp64
// atomic add per width.
#include <cuda_runtime_api.h>

#include <cstdio>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kCalibWarps = 8;
constexpr int kMaxWidths = 8;
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23: x + magic rounds x to an integer

struct CalibParams {
  const uint16_t* x;      // bf16 [T][hkv][D]
  long long T;
  int hkv;
  int nb;                 // Hadamard block
  int W;                  // widths
  int widths[kMaxWidths];
  double* out;            // [hkv][W]
  double scale;           // 1 / (nb * T * D)
};

template <int D>
__global__ void __launch_bounds__(kCalibWarps * 32)
    distortion_kernel(const __grid_constant__ CalibParams p) {
  constexpr int F = D / 16;   // elements per lane
  const int lane = threadIdx.x & 31, half = lane >> 4, l = lane & 15;
  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.y;
  double acc[kMaxWidths];     // this half-warp's squared errors, per width
#pragma unroll
  for (int w = 0; w < kMaxWidths; ++w) acc[w] = 0.0;

  const long long stride = static_cast<long long>(gridDim.x) * kCalibWarps * 2;
  for (long long t0 = (static_cast<long long>(blockIdx.x) * kCalibWarps + warp) * 2; t0 < p.T;
       t0 += stride) {
    const long long t = t0 + half;
    const bool valid = t < p.T;     // the loop is warp-uniform; half 1 may be past the end
    float v[F];
    if (valid) {
      const uint16_t* row = p.x + (t * p.hkv + h) * D + F * l;
      if constexpr (F == 8) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(row);
        v[0] = bf16lo(w4.x); v[1] = bf16hi(w4.x); v[2] = bf16lo(w4.y); v[3] = bf16hi(w4.y);
        v[4] = bf16lo(w4.z); v[5] = bf16hi(w4.z); v[6] = bf16lo(w4.w); v[7] = bf16hi(w4.w);
      } else {
        const uint2 w2 = *reinterpret_cast<const uint2*>(row);
        v[0] = bf16lo(w2.x); v[1] = bf16hi(w2.x); v[2] = bf16lo(w2.y); v[3] = bf16hi(w2.y);
      }
    } else {
#pragma unroll
      for (int e = 0; e < F; ++e) v[e] = 0.f;
    }
    // unnormalised Sylvester transform of each block of nb elements: stages
    // inside the lane, then across the lanes of the half-warp (partner l ^ m)
#pragma unroll
    for (int hs = 1; hs < F; hs <<= 1) {
      if (hs < p.nb) {
#pragma unroll
        for (int e = 0; e < F; ++e) {
          if (!(e & hs)) {
            const float a = v[e], c = v[e + hs];
            v[e] = __fadd_rn(a, c);
            v[e + hs] = __fsub_rn(a, c);
          }
        }
      }
    }
    for (int m = 1; m * F < p.nb; m <<= 1) {
      const bool upper = l & m;
#pragma unroll
      for (int e = 0; e < F; ++e) {
        const float o = __shfl_xor_sync(kFullMask, v[e], m);
        v[e] = upper ? __fsub_rn(o, v[e]) : __fadd_rn(v[e], o);
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
    const float zf = __half2float(__float2half_rd(mn));
    const float span = __fsub_rn(mx, zf);
#pragma unroll
    for (int w = 0; w < kMaxWidths; ++w) {
      if (w >= p.W) break;
      const float M = static_cast<float>((1 << p.widths[w]) - 1);   // levels
      const float sf = __half2float(__float2half_ru(__fdiv_rn(span, M)));
      const float inv = sf > 0.f ? __frcp_rn(sf) : 0.f;
      float e2 = 0.f;
#pragma unroll
      for (int e = 0; e < F; ++e) {
        // round-half-even of the exact product (one rounding of product + magic)
        float c = __fsub_rn(__fmaf_rn(__fsub_rn(v[e], zf), inv, kRoundMagic), kRoundMagic);
        c = fminf(fmaxf(c, 0.f), M);
        const float d = __fsub_rn(v[e], __fmaf_rn(c, sf, zf));
        e2 = __fmaf_rn(d, d, e2);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) e2 += __shfl_xor_sync(kFullMask, e2, o);
      if (valid) acc[w] += static_cast<double>(e2);
    }
  }

  // CTA sums: lane 0 of each half-warp holds its sums; fixed-order reduction
  __shared__ double red[kCalibWarps * 2][kMaxWidths];
  if (l == 0) {
#pragma unroll
    for (int w = 0; w < kMaxWidths; ++w) red[warp * 2 + half][w] = acc[w];
  }
  __syncthreads();
  if (threadIdx.x < p.W) {
    double s = 0.0;
    for (int i = 0; i < kCalibWarps * 2; ++i) s += red[i][threadIdx.x];
    atomicAdd(p.out + h * p.W + threadIdx.x, s * p.scale);
  }
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_distortion(int head_dim, int had_block, int num_kv_heads, const void* X,
                                     long long T, const int* widths, int n_widths, double* mse,
                                     void* stream) {
  char msg[200];
  if (head_dim != 64 && head_dim != 128) {
    std::snprintf(msg, sizeof msg, "kvq_distortion: head_dim %d not built (64, 128)", head_dim);
    return kvq::set_last_error(KVQ_EUNSUPPORTED, msg);
  }
  if ((had_block != 1 && had_block != 32 && had_block != 64 && had_block != 128) ||
      head_dim % had_block) {
    std::snprintf(msg, sizeof msg,
                  "kvq_distortion: had_block %d must be 1, 32, 64 or 128 and divide %d",
                  had_block, head_dim);
    return kvq::set_last_error(KVQ_EINVAL, msg);
  }
  if (num_kv_heads < 1 || num_kv_heads > 65535)
    return kvq::set_last_error(KVQ_EINVAL, "kvq_distortion: num_kv_heads must be 1 .. 65535");
  if (T < 0) return kvq::set_last_error(KVQ_EINVAL, "kvq_distortion: T must be >= 0");
  if (!widths || n_widths < 1 || n_widths > kvq::kMaxWidths)
    return kvq::set_last_error(KVQ_EINVAL, "kvq_distortion: n_widths must be 1 .. 8 with widths");
  kvq::CalibParams p;
  for (int w = 0; w < n_widths; ++w) {
    if (widths[w] < 1 || widths[w] > 8) {
      std::snprintf(msg, sizeof msg, "kvq_distortion: width %d outside 1 .. 8", widths[w]);
      return kvq::set_last_error(KVQ_EINVAL, msg);
    }
    p.widths[w] = widths[w];
  }
  for (int w = n_widths; w < kvq::kMaxWidths; ++w) p.widths[w] = 1;
  if (!mse || reinterpret_cast<uintptr_t>(mse) % 8)
    return kvq::set_last_error(KVQ_EINVAL, "kvq_distortion: mse must be non-NULL and 8-byte aligned");
  if (T > 0 && (!X || reinterpret_cast<uintptr_t>(X) % 16))
    return kvq::set_last_error(KVQ_EINVAL, "kvq_distortion: X must be non-NULL and 16-byte aligned");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(mse, 0, sizeof(double) * num_kv_heads * n_widths, s);
  if (e == cudaSuccess && T > 0) {
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) {
      p.x = static_cast<const uint16_t*>(X);
      p.T = T;
      p.hkv = num_kv_heads;
      p.nb = had_block;
      p.W = n_widths;
      p.out = mse;
      p.scale = 1.0 / (static_cast<double>(had_block) * static_cast<double>(T) * head_dim);
      // about 8 CTAs of 8 warps per SM over all heads, at least one per head
      const long long per_cta = kvq::kCalibWarps * 2;
      long long g = (T + per_cta - 1) / per_cta;
      const long long cap = (8LL * sms + num_kv_heads - 1) / num_kv_heads;
      if (g > cap) g = cap;
      if (g < 1) g = 1;
      const dim3 grid(static_cast<unsigned>(g), static_cast<unsigned>(num_kv_heads));
      if (head_dim == 128)
        kvq::distortion_kernel<128><<<grid, kvq::kCalibWarps * 32, 0, s>>>(p);
      else
        kvq::distortion_kernel<64><<<grid, kvq::kCalibWarps * 32, 0, s>>>(p);
      e = cudaGetLastError();
    }
  }
  if (e != cudaSuccess) {
    std::snprintf(msg, sizeof msg, "kvq_distortion: %s", cudaGetErrorString(e));
    return kvq::set_last_error(KVQ_ECUDA, msg);
  }
  return KVQ_OK;
}
