// fwd_f32_simt.cu -- exact fp32 tiled attention forward on CUDA cores.
//
// Same computation as the tensor-core kernel ("Flash attention and efficient
// attention -- Hinglish notes", "The Standard Attention Problem", evaluated
// with the running maximum / running sum of "Derivation: Incremental
// Softmax", Steps 1-3), in plain fp32 with the accurate expf/logf so that
// results stay within 1e-5 of the float64 definition; TF32 tensor cores could
// not meet that bound.
//
// One warp per query row.  Keys are visited in tiles of 32: lane t scores key
// (tile start + t); the tile's maximum and the sum of its exponentials are
// combined across the warp with shuffles; each lane then accumulates the
// output dimensions t, t+32, t+64, t+96 over the tile's keys, rescaling its
// partial sums when the running maximum rises.
#include <cmath>

#include "kernels.h"

namespace fa {
namespace {

constexpr int kWarpsPerBlock = 4;
constexpr int kMaxD = 128;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    fa_fwd_f32_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                           float* __restrict__ o, float* __restrict__ lse, long long rows, int N, int d,
                           int window_r, float scale) {
  __shared__ float sq[kWarpsPerBlock][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  if (row >= rows) return;  // whole warp leaves together
  const long long bh = row / N;
  const int i = static_cast<int>(row % N);
  const float* qr = q + row * d;
  const float* kh = k + bh * static_cast<long long>(N) * d;
  const float* vh = v + bh * static_cast<long long>(N) * d;
  for (int c = lane; c < d; c += 32) sq[warp][c] = qr[c];
  __syncwarp();

  int lo = 0, hi = N;
  if (window_r >= 0) {
    lo = max(0, i - window_r);
    hi = min(N, i + window_r + 1);
  }
  float m = -INFINITY, l = 0.f;
  float acc[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
  for (int j0 = lo; j0 < hi; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < hi) {
      const float* kr = kh + static_cast<long long>(j) * d;
      float dot = 0.f;
      for (int c = 0; c < d; ++c) dot = fmaf(sq[warp][c], kr[c], dot);
      s = dot * scale;
    }
    const float m_new = fmaxf(m, warp_max(s));  // finite: key j0 is always in range
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float pj = (j < hi) ? expf(s - m_new) : 0.f;
    l = l * alpha + warp_sum(pj);
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) acc[t] *= alpha;
    const int cnt = min(32, hi - j0);
    for (int jj = 0; jj < cnt; ++jj) {
      const float pb = __shfl_sync(0xffffffffu, pj, jj);
      const float* vr = vh + static_cast<long long>(j0 + jj) * d;
#pragma unroll
      for (int t = 0; t < kMaxD / 32; ++t) {
        const int c = lane + 32 * t;
        if (c < d) acc[t] = fmaf(pb, vr[c], acc[t]);
      }
    }
    m = m_new;
  }
  float* orow = o + row * d;
#pragma unroll
  for (int t = 0; t < kMaxD / 32; ++t) {
    const int c = lane + 32 * t;
    if (c < d) orow[c] = acc[t] / l;
  }
  if (lse != nullptr && lane == 0) lse[row] = m + logf(l);
}

}  // namespace

cudaError_t launch_fwd_f32_simt(const FwdParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffffLL || p.d > kMaxD) return cudaErrorInvalidConfiguration;
  fa_fwd_f32_simt_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, s>>>(
      static_cast<const float*>(p.q), static_cast<const float*>(p.k), static_cast<const float*>(p.v),
      static_cast<float*>(p.o), p.lse, rows, p.N, p.d, p.window_r, p.scale);
  return cudaGetLastError();
}

}  // namespace fa
