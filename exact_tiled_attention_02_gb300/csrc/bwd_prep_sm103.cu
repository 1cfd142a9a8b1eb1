// bwd_prep_sm103.cu -- the element-wise kernels around the attention
// backward's main kernels (bf16, every head dimension), and its workspace.
//
// "Flash attention and efficient attention -- Hinglish notes", "Backward
// Pass: Recomputation": the backward rebuilds P from the forward's logsumexp;
// the per-row quantities it needs besides lse are computed here.  The
// gradient formulas are the derivative of the forward definition (the pages
// print none): D_i = sum_j P_ij dP_ij = sum_k dO_ik O_ik.
//
//   bwd_prep  per (padded) query row: -D_i and the lse term the main kernel
//             uses (-lse_i log2 e for d = 96 / 128; for d = 64, -lse_i / scale
//             and -D_i as three bf16 terms each, the operand rows that kernel's
//             tensor core adds in), and the row of the fp32 dQ accumulator
//             zeroed.  Rows are padded to a multiple of 128: padding rows get
//             D = 0 and a term that makes their P 0.  Blocks past the rows
//             zero the fp32 dV / dK partial rows of the split key tiles.
//   bwd_dq    dQ = bf16(scale * accumulator); blocks past it convert the
//             split key tiles' dV / dK partial sums to bf16.
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

__host__ __device__ __forceinline__ int npad128(int n) { return (n + 127) & ~127; }

// Three bf16 terms whose sum is x to fp32 precision (each term takes what the
// previous ones left; the differences are exact in fp32), with five zeros:
// one 16-byte row of a K = 16 operand whose other 8 elements are zero.
__device__ __forceinline__ uint4 bf16_split3_row(float x) {
  const __nv_bfloat16 h1 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h1);
  const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
  const __nv_bfloat16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
  uint4 v;
  v.x = static_cast<uint32_t>(__bfloat16_as_ushort(h1)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h2)) << 16);
  v.y = static_cast<uint32_t>(__bfloat16_as_ushort(h3));
  v.z = 0u;
  v.w = 0u;
  return v;
}

// Lane groups of G = 8 (d = 64) or 16 (d = 96, 128) lanes per row, lane c of
// a group holding the 16-byte chunk c (8 bf16) of O and of dO; a warp covers
// 32 / G rows per pass and U = 4 passes, with every load of the four passes
// issued before any is used, so that each SM has enough bytes in flight to
// keep HBM busy.  A warp's rows are consecutive padded rows of one (batch,
// head): np is a multiple of 128 and a warp's row count divides 128.
template <int D>
struct PrepShape {
  static constexpr int CH = D / 8;                          // 16-byte chunks per row
  static constexpr int G = CH <= 8 ? 8 : (CH <= 16 ? 16 : 32);  // lanes per row
  static constexpr int RPW = 32 / G;                        // rows per warp and pass
  static constexpr int U = 4;                               // passes per warp
  static constexpr int RW = RPW * U;                        // rows per warp
  static constexpr int RB = 8 * RW;                         // rows per 256-thread block
  static_assert(128 % RW == 0, "a warp's rows stay within one (batch, head)");
};

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ lse2,
                                                         float* __restrict__ dsum, float* __restrict__ dq_acc, int BH,
                                                         int N, float inv_scale, long long row_blocks,
                                                         float* __restrict__ kv_part, long long part4) {
  using S = PrepShape<D>;
  constexpr bool kSplit = D == 64;  // the d = 64 kernel's three-term operand rows
  if (blockIdx.x >= row_blocks) {
    // zero the split tiles' partial rows, one float4 per thread
    const long long i = (static_cast<long long>(blockIdx.x) - row_blocks) * 256 + threadIdx.x;
    if (i < part4) reinterpret_cast<float4*>(kv_part)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int np = npad128(N);
  const long long base = (static_cast<long long>(blockIdx.x) * 8 + warp) * S::RW;  // first padded row of the warp
  if (base >= static_cast<long long>(BH) * np) return;  // the warp's rows all lie past the end
  const long long bh = base / np;
  const int i0 = static_cast<int>(base - bh * np);
  const int c = lane % S::G, sub = lane / S::G;
  const bool lane_on = c < S::CH;
  uint4 ov[S::U], gv[S::U];
  float lv[S::U];
#pragma unroll
  for (int u = 0; u < S::U; ++u) {
    const int i = i0 + u * S::RPW + sub;
    ov[u] = gv[u] = make_uint4(0u, 0u, 0u, 0u);
    lv[u] = 0.f;
    if (lane_on && i < N) {
      const long long src = (bh * N + i) * D + 8 * c;
      ov[u] = __ldg(reinterpret_cast<const uint4*>(o + src));
      gv[u] = __ldg(reinterpret_cast<const uint4*>(dO + src));
      if (c == 0) lv[u] = __ldg(lse + bh * N + i);
    }
  }
#pragma unroll
  for (int u = 0; u < S::U; ++u) {
    const int i = i0 + u * S::RPW + sub;
    if (lane_on && i < N) {
      float4* z = reinterpret_cast<float4*>(dq_acc + (bh * N + i) * D + 8 * c);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int u = 0; u < S::U; ++u) {
    const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&ov[u]);
    const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&gv[u]);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __bfloat1622float2(op[e]);
      const float2 b = __bfloat1622float2(gp[e]);
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
#pragma unroll
    for (int sft = S::G / 2; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
    const int i = i0 + u * S::RPW + sub;
    if (c == 0) {
      const long long row = bh * np + i;  // padded row index
      if (kSplit) {
        // padding rows: -lse / scale far below any logit, so their P underflows to 0
        reinterpret_cast<uint4*>(lse2)[row] = bf16_split3_row(i < N ? -lv[u] * inv_scale : -1e30f);
        reinterpret_cast<uint4*>(dsum)[row] = bf16_split3_row(i < N ? -acc : 0.f);
      } else {
        lse2[row] = i < N ? -lv[u] * 1.4426950408889634f : -INFINITY;
        dsum[row] = i < N ? -acc : 0.f;
      }
    }
  }
}

// dQ = bf16(scale * acc), 8 elements per thread; threads past the n8 groups
// of dQ convert the split key tiles' partial rows (already scaled) into dV
// and dK, 8 elements each
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                       long long n8, float scale, const float* __restrict__ kv_part,
                                                       __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                                                       int n_full, int n_split, int N, int d) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) {
    const int c8n = d / 8;                          // 8-element groups per row
    const long long per = 128LL * c8n;              // groups per (tile, dV or dK)
    const long long u = i - n8;
    if (u >= 2 * per * n_split) return;
    const int s = static_cast<int>(u / (2 * per));  // split tile
    const int which = static_cast<int>((u / per) & 1);
    const int row = static_cast<int>((u % per) / c8n), c8 = static_cast<int>(u % c8n);
    const int nkt = (N + 127) / 128;
    const int tile = n_full + s;
    const long long bh = tile / nkt;
    const int kr = (tile % nkt) * 128 + row;
    if (kr >= N) return;
    const float4* src = reinterpret_cast<const float4*>(kv_part + u * 8);
    const float4 a = src[0], b = src[1];
    uint4 out;
    out.x = pack_bf16x2(a.x, a.y);
    out.y = pack_bf16x2(a.z, a.w);
    out.z = pack_bf16x2(b.x, b.y);
    out.w = pack_bf16x2(b.z, b.w);
    __nv_bfloat16* dst = which == 0 ? dv : dk;
    *reinterpret_cast<uint4*>(dst + (bh * N + kr) * d + 8 * c8) = out;
    return;
  }
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16x2(a.x * scale, a.y * scale);
  out.y = pack_bf16x2(a.z * scale, a.w * scale);
  out.z = pack_bf16x2(b.x * scale, b.y * scale);
  out.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = out;
}

}  // namespace

size_t bwd_workspace_layout(int BH, int N, int d, size_t* off_lse2, size_t* off_dsum, size_t* off_part) {
  const size_t rows = static_cast<size_t>(BH) * N;
  const size_t prow = static_cast<size_t>(BH) * npad128(N);
  const size_t acc = (rows * d * sizeof(float) + 255) & ~size_t(255);
  // d = 64 stores each row's value as three bf16 terms in a 16-byte row
  const size_t vec = (prow * (d == 64 ? 16 : sizeof(float)) + 255) & ~size_t(255);
  // bf16 head dimensions: fp32 dV and dK rows of up to kMaxSplitTiles split key tiles
  const size_t tiles = static_cast<size_t>(BH) * ((N + 127) / 128);
  const size_t split = (d == 64 || d == 96 || d == 128) ? (tiles < kMaxSplitTiles ? tiles : kMaxSplitTiles) : 0;
  const size_t part = split * 2 * 128 * d * sizeof(float);  // a multiple of 256
  if (off_lse2) *off_lse2 = acc;
  if (off_dsum) *off_dsum = acc + vec;
  if (off_part) *off_part = acc + 2 * vec;
  return acc + 2 * vec + part;
}

cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.BH) * npad128(p.N);
  const int rb = p.d == 64 ? PrepShape<64>::RB : PrepShape<128>::RB;
  static_assert(PrepShape<96>::RB == PrepShape<128>::RB, "d = 96 and 128 share a block shape");
  const long long row_blocks = (rows + rb - 1) / rb;
  const long long part4 = static_cast<long long>(p.n_split) * 2 * 128 * p.d / 4;
  const long long blocks = row_blocks + (part4 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const auto o = static_cast<const __nv_bfloat16*>(p.o);
  const auto dO = static_cast<const __nv_bfloat16*>(p.dO);
  const unsigned g = static_cast<unsigned>(blocks);
  const float inv = 1.f / p.scale;
  if (p.d == 64)
    fa_bwd_prep_kernel<64><<<g, 256, 0, s>>>(o, dO, p.lse, p.lse2, p.dsum, p.dq_acc, p.BH, p.N, inv, row_blocks,
                                             p.kv_part, part4);
  else if (p.d == 96)
    fa_bwd_prep_kernel<96><<<g, 256, 0, s>>>(o, dO, p.lse, p.lse2, p.dsum, p.dq_acc, p.BH, p.N, inv, row_blocks,
                                             p.kv_part, part4);
  else if (p.d == 128)
    fa_bwd_prep_kernel<128><<<g, 256, 0, s>>>(o, dO, p.lse, p.lse2, p.dsum, p.dq_acc, p.BH, p.N, inv, row_blocks,
                                              p.kv_part, part4);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdParams& p, cudaStream_t s) {
  const long long n8 = static_cast<long long>(p.BH) * p.N * p.d / 8;
  const long long total = n8 + static_cast<long long>(p.n_split) * 2 * 128 * p.d / 8;
  if ((total + 255) / 256 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_bwd_dq_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, s>>>(
      p.dq_acc, static_cast<__nv_bfloat16*>(p.dq), n8, p.scale, p.kv_part, static_cast<__nv_bfloat16*>(p.dk),
      static_cast<__nv_bfloat16*>(p.dv), p.n_full, p.n_split, p.N, p.d);
  return cudaGetLastError();
}

}  // namespace fa
