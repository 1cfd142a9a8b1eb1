// bwd_f32_simt.cu -- exact fp32 attention backward on CUDA cores.
//
// The same recomputation as the bf16 tensor-core backward ("Flash attention
// and efficient attention -- Hinglish notes", "Backward Pass: Recomputation":
// P is rebuilt from Q, K and the forward's logsumexp, never read), in plain
// fp32 with the accurate expf so that the gradients stay close to the float64
// derivative.  Formulas (the derivative of the forward definition; the pages
// print none):  P_ij = exp(scale q_i.k_j - lse_i),  dP_ij = dO_i.v_j,
// D_i = sum_k dO_ik O_ik,  dS_ij = P_ij (dP_ij - D_i),
// dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
// dV_j = sum_i P_ij dO_i.
//
// Three kernels, one warp per row each, no atomics (bitwise repeatable):
//   prep    D_i into the workspace;
//   dq      one warp per query row i: lane t recomputes P and dS for key
//           (tile start + t) of a 32-key tile; each lane then accumulates
//           dQ_i's dimensions t, t+32, t+64, t+96 over the tile's keys;
//   dkdv    one warp per key row j, the mirror image over 32-query tiles.
// With a window of radius r, row i visits only keys |i - j| <= r and key j
// only such queries, which is exactly where P is non-zero.
#include <cmath>

#include "kernels.h"

namespace fa {
namespace {

constexpr int kWarpsPerBlock = 4;
constexpr int kMaxD = 128;
constexpr int kPerLane = kMaxD / 32;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// dot(a, b) over d elements: a in shared memory (the warp's own row), b in
// global memory (a different row per lane).
__device__ __forceinline__ float dot_row(const float* a, const float* __restrict__ b, int d) {
  float acc = 0.f;
  for (int c = 0; c < d; ++c) acc = fmaf(a[c], b[c], acc);
  return acc;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    fa_bwd_f32_prep_kernel(const float* __restrict__ o, const float* __restrict__ dO, float* __restrict__ dsum,
                           long long rows, int d) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  if (row >= rows) return;
  const float* orow = o + row * d;
  const float* grow = dO + row * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc = fmaf(orow[c], grow[c], acc);
  acc = warp_sum(acc);
  if (lane == 0) dsum[row] = acc;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    fa_bwd_f32_dq_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                         const float* __restrict__ lse, const float* __restrict__ dO,
                         const float* __restrict__ dsum, float* __restrict__ dq, long long rows, int N, int d,
                         int window_r, float scale) {
  __shared__ float sq[kWarpsPerBlock][kMaxD];
  __shared__ float sg[kWarpsPerBlock][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  if (row >= rows) return;  // whole warp leaves together
  const long long bh = row / N;
  const int i = static_cast<int>(row % N);
  const float* kh = k + bh * static_cast<long long>(N) * d;
  const float* vh = v + bh * static_cast<long long>(N) * d;
  for (int c = lane; c < d; c += 32) {
    sq[warp][c] = q[row * d + c];
    sg[warp][c] = dO[row * d + c];
  }
  __syncwarp();
  const float lse_i = lse[row], D_i = dsum[row];

  int lo = 0, hi = N;
  if (window_r >= 0) {
    lo = max(0, i - window_r);
    hi = min(N, i + window_r + 1);
  }
  float acc[kPerLane] = {0.f, 0.f, 0.f, 0.f};
  for (int j0 = lo; j0 < hi; j0 += 32) {
    const int j = j0 + lane;
    float ds = 0.f;
    if (j < hi) {
      const float p = expf(dot_row(sq[warp], kh + static_cast<long long>(j) * d, d) * scale - lse_i);
      const float dp = dot_row(sg[warp], vh + static_cast<long long>(j) * d, d);
      ds = p * (dp - D_i);
    }
    const int cnt = min(32, hi - j0);
    for (int jj = 0; jj < cnt; ++jj) {
      const float db = __shfl_sync(0xffffffffu, ds, jj);
      const float* kr = kh + static_cast<long long>(j0 + jj) * d;
#pragma unroll
      for (int t = 0; t < kPerLane; ++t) {
        const int c = lane + 32 * t;
        if (c < d) acc[t] = fmaf(db, kr[c], acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kPerLane; ++t) {
    const int c = lane + 32 * t;
    if (c < d) dq[row * d + c] = acc[t] * scale;
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    fa_bwd_f32_dkdv_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                           const float* __restrict__ lse, const float* __restrict__ dO,
                           const float* __restrict__ dsum, float* __restrict__ dk, float* __restrict__ dv,
                           long long rows, int N, int d, int window_r, float scale) {
  __shared__ float sk[kWarpsPerBlock][kMaxD];
  __shared__ float sv[kWarpsPerBlock][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  if (row >= rows) return;
  const long long bh = row / N;
  const int j = static_cast<int>(row % N);
  const long long head = bh * static_cast<long long>(N);
  const float* qh = q + head * d;
  const float* gh = dO + head * d;
  for (int c = lane; c < d; c += 32) {
    sk[warp][c] = k[row * d + c];
    sv[warp][c] = v[row * d + c];
  }
  __syncwarp();

  int lo = 0, hi = N;
  if (window_r >= 0) {
    lo = max(0, j - window_r);
    hi = min(N, j + window_r + 1);
  }
  float acc_k[kPerLane] = {0.f, 0.f, 0.f, 0.f};
  float acc_v[kPerLane] = {0.f, 0.f, 0.f, 0.f};
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    float p = 0.f, ds = 0.f;
    if (i < hi) {
      p = expf(dot_row(sk[warp], qh + static_cast<long long>(i) * d, d) * scale - lse[head + i]);
      const float dp = dot_row(sv[warp], gh + static_cast<long long>(i) * d, d);
      ds = p * (dp - dsum[head + i]);
    }
    const int cnt = min(32, hi - i0);
    for (int ii = 0; ii < cnt; ++ii) {
      const float pb = __shfl_sync(0xffffffffu, p, ii);
      const float db = __shfl_sync(0xffffffffu, ds, ii);
      const float* qr = qh + static_cast<long long>(i0 + ii) * d;
      const float* gr = gh + static_cast<long long>(i0 + ii) * d;
#pragma unroll
      for (int t = 0; t < kPerLane; ++t) {
        const int c = lane + 32 * t;
        if (c < d) {
          acc_v[t] = fmaf(pb, gr[c], acc_v[t]);
          acc_k[t] = fmaf(db, qr[c], acc_k[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kPerLane; ++t) {
    const int c = lane + 32 * t;
    if (c < d) {
      dk[row * d + c] = acc_k[t] * scale;
      dv[row * d + c] = acc_v[t];
    }
  }
}

}  // namespace

cudaError_t launch_bwd_f32_simt(const BwdParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffffLL || p.d > kMaxD) return cudaErrorInvalidConfiguration;
  const unsigned grid = static_cast<unsigned>(blocks);
  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);
  const float* dO = static_cast<const float*>(p.dO);
  // D_i uses the workspace's D section as a plain [B*H*N] array
  fa_bwd_f32_prep_kernel<<<grid, kWarpsPerBlock * 32, 0, s>>>(static_cast<const float*>(p.o), dO, p.dsum, rows,
                                                               p.d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_f32_dq_kernel<<<grid, kWarpsPerBlock * 32, 0, s>>>(q, k, v, p.lse, dO, p.dsum, static_cast<float*>(p.dq),
                                                             rows, p.N, p.d, p.window_r, p.scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_f32_dkdv_kernel<<<grid, kWarpsPerBlock * 32, 0, s>>>(q, k, v, p.lse, dO, p.dsum,
                                                               static_cast<float*>(p.dk), static_cast<float*>(p.dv),
                                                               rows, p.N, p.d, p.window_r, p.scale);
  return cudaGetLastError();
}

}  // namespace fa
