// fwd_f32_simt.cu -- exact fp32 tiled attention forward on CUDA cores.
//
// Same computation as the tensor-core kernel ("Flash attention and efficient
// attention -- Hinglish notes", "The Standard Attention Problem", evaluated
// with the running maximum / running sum of "Derivation: Incremental
// Softmax", Steps 1-3), in plain fp32 with the accurate expf/logf so that
// results stay within 1e-5 of the float64 definition; TF32 tensor cores could
// not meet that bound.
//
// One CTA of 256 threads per 64 query rows of one (batch, head); key tiles of
// 64.  Q and each K tile sit in shared memory transposed ([d][64], so that
// four consecutive rows of one column are one 16-byte load), V row-major and
// P row-major.  Thread (ty, tx) = (tid / 16, tid % 16) owns query rows
// 4ty..4ty+3: it computes their scores against keys 4tx..4tx+3 (a 4 x 4
// register block, two 16-byte loads per 16 FMAs), and accumulates their
// output columns 4tx..4tx+3 and 64+4tx..64+4tx+3.  The 16 threads of one ty
// are one half-warp, so the row maximum and row sum of a tile take four
// shuffles each.  Head dimensions that are not a multiple of 4 are padded
// with zeros in shared memory.
#include <cmath>

#include "kernels.h"

namespace fa {
namespace {

constexpr int BQ = 64;        // query rows per CTA
constexpr int BK = 64;        // keys per tile
constexpr int kThreads = 256;
constexpr int kMaxD = 128;
// shared memory for head dimensions up to DR (Qt, Kt, Vs, Ps): 112 KB at
// DR = 128 (two CTAs per SM), 64 KB at DR = 64 (three)
template <int DR>
constexpr int smem_bytes() {
  return (DR * BQ + DR * BK + BK * DR + BQ * BK) * 4;
}

__device__ __forceinline__ float half_warp_max(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float half_warp_sum(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// rows [r0, r0 + 64) of a [N][d] matrix into shared memory: transposed
// (dst[c][row], 64 floats per c) or row-major (dst[row][c], ldr floats per
// row), columns up to dp (d rounded up to 4), zero past N and past d
template <bool TRANSPOSE>
__device__ __forceinline__ void load_tile(float* dst, const float* __restrict__ src, int r0, int N, int d, int dp,
                                          int ldr) {
  const int tid = threadIdx.x;
  if ((d & 3) == 0) {
    const int c4n = dp >> 2;
    for (int idx = tid; idx < 64 * c4n; idx += kThreads) {
      const int row = idx & 63, c4 = idx >> 6;  // consecutive threads, consecutive rows
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r0 + row < N) v = *reinterpret_cast<const float4*>(src + static_cast<long long>(r0 + row) * d + 4 * c4);
      if (TRANSPOSE) {
        dst[(4 * c4 + 0) * 64 + row] = v.x;
        dst[(4 * c4 + 1) * 64 + row] = v.y;
        dst[(4 * c4 + 2) * 64 + row] = v.z;
        dst[(4 * c4 + 3) * 64 + row] = v.w;
      } else {
        *reinterpret_cast<float4*>(dst + row * ldr + 4 * c4) = v;
      }
    }
  } else {
    for (int idx = tid; idx < 64 * dp; idx += kThreads) {
      const int row = idx & 63, c = idx >> 6;
      const float v = (r0 + row < N && c < d) ? src[static_cast<long long>(r0 + row) * d + c] : 0.f;
      if (TRANSPOSE)
        dst[c * 64 + row] = v;
      else
        dst[row * ldr + c] = v;
    }
  }
}

template <bool HI>  // output columns 64.. exist (d > 64)
__global__ void __launch_bounds__(kThreads, HI ? 2 : 3)
    fa_fwd_f32_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                           float* __restrict__ o, float* __restrict__ lse, int N, int d, int window_r, float scale) {
  constexpr int DR = HI ? kMaxD : 64;  // head-dimension extent of the tiles
  constexpr int M = HI ? 8 : 4;        // output columns per thread
  extern __shared__ float4 smem4[];
  float* Qt = reinterpret_cast<float*>(smem4);  // [DR][64]
  float* Kt = Qt + DR * BQ;                     // [DR][64]
  float* Vs = Kt + DR * BK;                     // [64][DR]
  float* Ps = Vs + BK * DR;                     // [64][64]
  const int nqt = (N + BQ - 1) / BQ;
  const long long bh = blockIdx.x / nqt;
  const int q0 = (blockIdx.x % nqt) * BQ;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int dp = (d + 3) & ~3;
  const long long head = bh * static_cast<long long>(N) * d;
  const float* qh = q + head;
  const float* kh = k + head;
  const float* vh = v + head;

  load_tile<true>(Qt, qh, q0, N, d, dp, DR);

  int j_lo = 0, j_hi = N;  // keys that some row of this CTA sees
  if (window_r >= 0) {
    j_lo = max(0, q0 - window_r);
    j_hi = min(N, q0 + BQ - 1 + window_r + 1);
  }
  float m[4], l[4], acc[4][M];
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    m[ii] = -INFINITY;
    l[ii] = 0.f;
#pragma unroll
    for (int c = 0; c < M; ++c) acc[ii][c] = 0.f;
  }
  for (int k0 = (j_lo / BK) * BK; k0 < j_hi; k0 += BK) {
    __syncthreads();  // the previous tile's K, V and P are no longer read
    load_tile<true>(Kt, kh, k0, N, d, dp, DR);
    load_tile<false>(Vs, vh, k0, N, d, dp, DR);
    __syncthreads();
    // ---- S = Q K^T for rows 4ty.., keys 4tx..
    float s[4][4];
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) s[ii][jj] = 0.f;
#pragma unroll 4
    for (int c = 0; c < dp; ++c) {
      const float4 a = *reinterpret_cast<const float4*>(Qt + c * 64 + 4 * ty);
      const float4 b = *reinterpret_cast<const float4*>(Kt + c * 64 + 4 * tx);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) s[ii][jj] = fmaf(av[ii], bv[jj], s[ii][jj]);
    }
    // ---- scale, mask, online softmax (per row: max and sum over the half-warp)
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int i = q0 + 4 * ty + ii;
      float tmax = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = k0 + 4 * tx + jj;
        const bool in = j < N && (window_r < 0 || (j >= i - window_r && j <= i + window_r));
        s[ii][jj] = in ? s[ii][jj] * scale : -INFINITY;
        tmax = fmaxf(tmax, s[ii][jj]);
      }
      const float m_new = fmaxf(m[ii], half_warp_max(tmax));
      const float alpha = (m[ii] == -INFINITY) ? 0.f : expf(m[ii] - m_new);
      float rs = 0.f;
      float pv[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        pv[jj] = (s[ii][jj] == -INFINITY) ? 0.f : expf(s[ii][jj] - m_new);
        rs += pv[jj];
      }
      l[ii] = l[ii] * alpha + half_warp_sum(rs);
      m[ii] = m_new;
#pragma unroll
      for (int c = 0; c < M; ++c) acc[ii][c] *= alpha;
      *reinterpret_cast<float4*>(Ps + (4 * ty + ii) * BK + 4 * tx) = make_float4(pv[0], pv[1], pv[2], pv[3]);
    }
    __syncthreads();
    // ---- O += P V for rows 4ty.., columns 4tx.. and 64 + 4tx..
#pragma unroll 2
    for (int k4 = 0; k4 < BK; k4 += 4) {
      float p[4][4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const float4 t = *reinterpret_cast<const float4*>(Ps + (4 * ty + ii) * BK + k4);
        p[ii][0] = t.x;
        p[ii][1] = t.y;
        p[ii][2] = t.z;
        p[ii][3] = t.w;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 v0 = *reinterpret_cast<const float4*>(Vs + (k4 + kk) * DR + 4 * tx);
        const float vv0[4] = {v0.x, v0.y, v0.z, v0.w};
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[ii][c] = fmaf(p[ii][kk], vv0[c], acc[ii][c]);
        if constexpr (HI) {
          const float4 v1 = *reinterpret_cast<const float4*>(Vs + (k4 + kk) * DR + 64 + 4 * tx);
          const float vv1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int ii = 0; ii < 4; ++ii)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[ii][4 + c] = fmaf(p[ii][kk], vv1[c], acc[ii][4 + c]);
        }
      }
    }
  }
  // ---- O / l and lse = m + ln l (natural log of the sum over scaled scores)
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int i = q0 + 4 * ty + ii;
    if (i >= N) continue;
    const float inv = 1.f / l[ii];
    float* orow = o + head + static_cast<long long>(i) * d;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (4 * tx + c < d) orow[4 * tx + c] = acc[ii][c] * inv;
      if constexpr (HI)
        if (64 + 4 * tx + c < d) orow[64 + 4 * tx + c] = acc[ii][4 + c] * inv;
    }
    if (lse != nullptr && tx == 0) lse[bh * N + i] = m[ii] + logf(l[ii]);
  }
}

}  // namespace

namespace {

template <bool HI>
cudaError_t launch_hi(const FwdParams& p, long long blocks, cudaStream_t s) {
  constexpr int SMEM = smem_bytes<HI ? kMaxD : 64>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_f32_simt_kernel<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  fa_fwd_f32_simt_kernel<HI><<<static_cast<unsigned>(blocks), kThreads, SMEM, s>>>(
      static_cast<const float*>(p.q), static_cast<const float*>(p.k), static_cast<const float*>(p.v),
      static_cast<float*>(p.o), p.lse, p.N, p.d, p.window_r, p.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32_simt(const FwdParams& p, cudaStream_t s) {
  if (p.d > kMaxD || p.d < 1) return cudaErrorInvalidConfiguration;
  const long long blocks = static_cast<long long>(p.BH) * ((p.N + BQ - 1) / BQ);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return ((p.d + 3) & ~3) > 64 ? launch_hi<true>(p, blocks, s) : launch_hi<false>(p, blocks, s);
}

}  // namespace fa
