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
// Three kernels, no atomics (bitwise repeatable):
//   prep    D_i into the workspace, one warp per row;
//   dkdv    one CTA of 256 threads per 64 keys of one head, over the 64-row
//           query tiles that can see them: S^T and dP^T as 4 x 4 register
//           blocks (thread (ty, tx): keys 4ty.., queries 4tx..), P^T and dS^T
//           through shared memory, then dV and dK for keys 4ty.. and head
//           columns tx, tx + 16, ... (eight per thread);
//   dq      the mirror image: one CTA per 64 queries over the key tiles,
//           S and dP as 4 x 4 blocks (queries 4ty.., keys 4tx..), dS through
//           shared memory, dQ for queries 4ty.. and columns tx, tx + 16, ...
// The streamed operand tiles sit in shared memory transposed ([d][64]), so
// that four rows of one column are one 16-byte load; the tiles that are also
// read one column at a time have 68-float rows, which spreads those loads
// over the banks (at most two threads of a half-warp share one).  Head
// dimensions that are not a multiple of 4 are padded with zeros.  With a
// window of radius r each tile loop visits only the tiles in the band, and
// the masked pairs get P = 0.
#include <cmath>

#include "kernels.h"

namespace fa {
namespace {

constexpr int kPrepWarps = 4;
constexpr int T = 64;          // rows per tile (keys or queries)
constexpr int kThreads = 256;
constexpr int kMaxD = 128;
constexpr int LD = 68;         // row stride (floats) of the tiles also read column-wise

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kPrepWarps * 32)
    fa_bwd_f32_prep_kernel(const float* __restrict__ o, const float* __restrict__ dO, float* __restrict__ dsum,
                           long long rows, int d) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kPrepWarps + warp;
  if (row >= rows) return;
  const float* orow = o + row * d;
  const float* grow = dO + row * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc = fmaf(orow[c], grow[c], acc);
  acc = warp_sum(acc);
  if (lane == 0) dsum[row] = acc;
}

// rows [r0, r0 + 64) of a [N][d] matrix into shared memory transposed:
// dst[c * ld + row] for c < dp (d rounded up to 4), zero past N and past d
__device__ __forceinline__ void load_t(float* dst, int ld, const float* __restrict__ src, int r0, int N, int d,
                                       int dp) {
  const int tid = threadIdx.x;
  if ((d & 3) == 0) {
    for (int idx = tid; idx < T * (dp >> 2); idx += kThreads) {
      const int row = idx & (T - 1), c4 = idx >> 6;  // consecutive threads, consecutive rows
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r0 + row < N) v = *reinterpret_cast<const float4*>(src + static_cast<long long>(r0 + row) * d + 4 * c4);
      dst[(4 * c4 + 0) * ld + row] = v.x;
      dst[(4 * c4 + 1) * ld + row] = v.y;
      dst[(4 * c4 + 2) * ld + row] = v.z;
      dst[(4 * c4 + 3) * ld + row] = v.w;
    }
  } else {
    for (int idx = tid; idx < T * dp; idx += kThreads) {
      const int row = idx & (T - 1), c = idx >> 6;
      dst[c * ld + row] = (r0 + row < N && c < d) ? src[static_cast<long long>(r0 + row) * d + c] : 0.f;
    }
  }
}

// 4 x 4 block of A B^T over c < dp: rows 4ty.. of A, rows 4tx.. of B, both
// stored transposed (a[c * lda + row])
__device__ __forceinline__ void block_abt(float (&acc)[4][4], const float* a, int lda, const float* b, int ldb, int dp,
                                          int ty, int tx) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int c = 0; c < dp; ++c) {
    const float4 x = *reinterpret_cast<const float4*>(a + c * lda + 4 * ty);
    const float4 y = *reinterpret_cast<const float4*>(b + c * ldb + 4 * tx);
    const float xv[4] = {x.x, x.y, x.z, x.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], yv[j], acc[i][j]);
  }
}

// acc[i][m] += sum_r w[(4ty + i) * T + r] * b[(tx + 16 m) * LD + r] over the
// 64 rows r of a tile: w row-major [64][64], b transposed with LD-float rows;
// M = 8 head-column slots (d up to 128) or 4 (d up to 64)
template <int M>
__device__ __forceinline__ void accum_wb(float (&acc)[4][M], const float* w, const float* b, int ty, int tx) {
#pragma unroll 2
  for (int r4 = 0; r4 < T; r4 += 4) {
    float wv[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t = *reinterpret_cast<const float4*>(w + (4 * ty + i) * T + r4);
      wv[i][0] = t.x;
      wv[i][1] = t.y;
      wv[i][2] = t.z;
      wv[i][3] = t.w;
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float bv = b[(tx + 16 * m) * LD + r4 + rr];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][m] = fmaf(wv[i][rr], bv, acc[i][m]);
      }
    }
  }
}

// shared memory of both tile kernels, in floats, for head dimensions up to
// DR (128, or 64: then two CTAs fit on an SM)
template <int DR>
constexpr int smem_bytes() {
  return (2 * DR * T + 2 * DR * LD + 2 * T * T) * 4;
}
static_assert(smem_bytes<64>() <= 113 * 1024, "two d <= 64 CTAs per SM");

// ---------------------------------------------------------------------------
// dK, dV: one CTA per 64 keys
// ---------------------------------------------------------------------------
template <bool HI>  // head columns 64.. exist (d > 64)
__global__ void __launch_bounds__(kThreads, HI ? 1 : 2)
    fa_bwd_f32_dkdv_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                           const float* __restrict__ lse, const float* __restrict__ dO,
                           const float* __restrict__ dsum, float* __restrict__ dk, float* __restrict__ dv, int N,
                           int d, int window_r, float scale) {
  constexpr int DR = HI ? kMaxD : 64;  // head-dimension rows of the transposed tiles
  constexpr int M = HI ? 8 : 4;        // head-column slots per thread
  extern __shared__ float4 smem4[];
  float* Kt = reinterpret_cast<float*>(smem4);  // [d][64]
  float* Vt = Kt + DR * T;                      // [d][64]
  float* Qt = Vt + DR * T;                      // [d][LD]
  float* Gt = Qt + DR * LD;                     // dO, [d][LD]
  float* Ps = Gt + DR * LD;                     // P^T [64 keys][64 queries]
  float* Ss = Ps + T * T;                       // dS^T [64 keys][64 queries]
  const int nkt = (N + T - 1) / T;
  const long long bh = blockIdx.x / nkt;
  const int k0 = (blockIdx.x % nkt) * T;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int dp = (d + 3) & ~3;
  const long long head = bh * static_cast<long long>(N) * d;
  load_t(Kt, T, k + head, k0, N, d, dp);
  load_t(Vt, T, v + head, k0, N, d, dp);
  int i_lo = 0, i_hi = N;  // queries that see some key of this tile
  if (window_r >= 0) {
    i_lo = max(0, k0 - window_r);
    i_hi = min(N, k0 + T - 1 + window_r + 1);
  }
  float acc_k[4][M], acc_v[4][M];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      acc_k[i][m] = 0.f;
      acc_v[i][m] = 0.f;
    }
  for (int q0 = (i_lo / T) * T; q0 < i_hi; q0 += T) {
    __syncthreads();  // the previous tile's Q, dO, P^T, dS^T are no longer read
    load_t(Qt, LD, q + head, q0, N, d, dp);
    load_t(Gt, LD, dO + head, q0, N, d, dp);
    __syncthreads();
    float s[4][4], g[4][4];
    block_abt(s, Kt, T, Qt, LD, dp, ty, tx);  // S^T: keys 4ty.., queries 4tx..
    block_abt(g, Vt, T, Gt, LD, dp, ty, tx);  // dP^T
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int i = q0 + 4 * tx + jj;
      const bool qok = i < N;
      const float l_i = qok ? lse[bh * N + i] : 0.f, d_i = qok ? dsum[bh * N + i] : 0.f;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int j = k0 + 4 * ty + ii;
        const bool in = qok && j < N && (window_r < 0 || (j >= i - window_r && j <= i + window_r));
        const float pij = in ? expf(s[ii][jj] * scale - l_i) : 0.f;
        s[ii][jj] = pij;
        g[ii][jj] = pij * (g[ii][jj] - d_i);
      }
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      *reinterpret_cast<float4*>(Ps + (4 * ty + ii) * T + 4 * tx) = make_float4(s[ii][0], s[ii][1], s[ii][2], s[ii][3]);
      *reinterpret_cast<float4*>(Ss + (4 * ty + ii) * T + 4 * tx) = make_float4(g[ii][0], g[ii][1], g[ii][2], g[ii][3]);
    }
    __syncthreads();
    accum_wb<M>(acc_v, Ps, Gt, ty, tx);  // dV += P^T dO
    accum_wb<M>(acc_k, Ss, Qt, ty, tx);  // dK += dS^T Q
  }
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int j = k0 + 4 * ty + ii;
    if (j >= N) continue;
    float* krow = dk + head + static_cast<long long>(j) * d;
    float* vrow = dv + head + static_cast<long long>(j) * d;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int c = tx + 16 * m;
      if (c < d) {
        krow[c] = acc_k[ii][m] * scale;
        vrow[c] = acc_v[ii][m];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// dQ: one CTA per 64 queries
// ---------------------------------------------------------------------------
template <bool HI>
__global__ void __launch_bounds__(kThreads, HI ? 1 : 2)
    fa_bwd_f32_dq_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                         const float* __restrict__ lse, const float* __restrict__ dO,
                         const float* __restrict__ dsum, float* __restrict__ dq, int N, int d, int window_r,
                         float scale) {
  constexpr int DR = HI ? kMaxD : 64;
  constexpr int M = HI ? 8 : 4;
  extern __shared__ float4 smem4[];
  float* Qt = reinterpret_cast<float*>(smem4);  // [d][64]
  float* Gt = Qt + DR * T;                      // dO, [d][64]
  float* Kt = Gt + DR * T;                      // [d][LD]
  float* Vt = Kt + DR * LD;                     // [d][LD]
  float* Ss = Vt + DR * LD;                     // dS [64 queries][64 keys]
  const int nqt = (N + T - 1) / T;
  const long long bh = blockIdx.x / nqt;
  const int q0 = (blockIdx.x % nqt) * T;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int dp = (d + 3) & ~3;
  const long long head = bh * static_cast<long long>(N) * d;
  load_t(Qt, T, q + head, q0, N, d, dp);
  load_t(Gt, T, dO + head, q0, N, d, dp);
  int j_lo = 0, j_hi = N;  // keys that some query of this tile sees
  if (window_r >= 0) {
    j_lo = max(0, q0 - window_r);
    j_hi = min(N, q0 + T - 1 + window_r + 1);
  }
  float l_i[4], d_i[4];
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int i = q0 + 4 * ty + ii;
    l_i[ii] = i < N ? lse[bh * N + i] : 0.f;
    d_i[ii] = i < N ? dsum[bh * N + i] : 0.f;
  }
  float acc[4][M];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[i][m] = 0.f;
  for (int k0 = (j_lo / T) * T; k0 < j_hi; k0 += T) {
    __syncthreads();  // the previous tile's K, V, dS are no longer read
    load_t(Kt, LD, k + head, k0, N, d, dp);
    load_t(Vt, LD, v + head, k0, N, d, dp);
    __syncthreads();
    float s[4][4], g[4][4];
    block_abt(s, Qt, T, Kt, LD, dp, ty, tx);  // S: queries 4ty.., keys 4tx..
    block_abt(g, Gt, T, Vt, LD, dp, ty, tx);  // dP
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int i = q0 + 4 * ty + ii;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = k0 + 4 * tx + jj;
        const bool in = i < N && j < N && (window_r < 0 || (j >= i - window_r && j <= i + window_r));
        const float pij = in ? expf(s[ii][jj] * scale - l_i[ii]) : 0.f;
        g[ii][jj] = pij * (g[ii][jj] - d_i[ii]);
      }
      *reinterpret_cast<float4*>(Ss + (4 * ty + ii) * T + 4 * tx) = make_float4(g[ii][0], g[ii][1], g[ii][2], g[ii][3]);
    }
    __syncthreads();
    accum_wb<M>(acc, Ss, Kt, ty, tx);  // dQ += dS K
  }
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int i = q0 + 4 * ty + ii;
    if (i >= N) continue;
    float* qrow = dq + head + static_cast<long long>(i) * d;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int c = tx + 16 * m;
      if (c < d) qrow[c] = acc[ii][m] * scale;
    }
  }
}

}  // namespace

namespace {

// the two tile kernels for head dimensions up to 64 (HI = false) or 128
template <bool HI>
cudaError_t launch_tiles(const BwdParams& p, long long tiles, cudaStream_t s) {
  constexpr int SMEM = smem_bytes<HI ? kMaxD : 64>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_f32_dkdv_kernel<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_bwd_f32_dq_kernel<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);
  const float* dO = static_cast<const float*>(p.dO);
  fa_bwd_f32_dq_kernel<HI><<<static_cast<unsigned>(tiles), kThreads, SMEM, s>>>(
      q, k, v, p.lse, dO, p.dsum, static_cast<float*>(p.dq), p.N, p.d, p.window_r, p.scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_f32_dkdv_kernel<HI><<<static_cast<unsigned>(tiles), kThreads, SMEM, s>>>(
      q, k, v, p.lse, dO, p.dsum, static_cast<float*>(p.dk), static_cast<float*>(p.dv), p.N, p.d, p.window_r,
      p.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_f32_simt(const BwdParams& p, cudaStream_t s) {
  if (p.d > kMaxD || p.d < 1) return cudaErrorInvalidConfiguration;
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const long long prep_blocks = (rows + kPrepWarps - 1) / kPrepWarps;
  const long long tiles = static_cast<long long>(p.BH) * ((p.N + T - 1) / T);
  if (prep_blocks > 0x7fffffffLL || tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // D_i uses the workspace's D section as a plain [B*H*N] array
  fa_bwd_f32_prep_kernel<<<static_cast<unsigned>(prep_blocks), kPrepWarps * 32, 0, s>>>(
      static_cast<const float*>(p.o), static_cast<const float*>(p.dO), p.dsum, rows, p.d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return ((p.d + 3) & ~3) > 64 ? launch_tiles<true>(p, tiles, s) : launch_tiles<false>(p, tiles, s);
}

}  // namespace fa
