// fwd_bf16_sm103.cu -- tiled exact attention forward, bf16 in / fp32
// accumulate, for GB300 (sm_103a): TMA + mbarrier ring, tcgen05.mma into
// tensor memory, online softmax on CUDA cores.
//
// What it computes: for each (batch, head) and query row i,
//   O_i = sum_j softmax_j(S_i) V_j,  S_ij = scale * q_i . k_j   (masked: -inf)
//   lse_i = ln sum_j exp(S_ij)
// following "Flash attention and efficient attention -- Hinglish notes",
// "The Standard Attention Problem", evaluated one key/value tile at a time
// with the running maximum / running sum merge of that page's "Derivation:
// Incremental Softmax" (Steps 1-3) and of "Compute attention one tile at a
// time" (TensorViz), step "tiles": the maximum and denominator of each query
// row are carried across tiles, earlier contributions are rescaled when the
// maximum rises, and the numerator is divided by the denominator once, at the
// end.  The score tile lives only in tensor memory; nothing of size N x N
// reaches device memory.
//
// CTA = one 128-row query tile of one (batch, head); 192 threads:
//   warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t)
//   warp  4    TMA producer (one elected lane)
//   warp  5    TMEM owner + tcgen05.mma issuer (one elected lane)
// Tensor memory (512 columns x 128 lanes, fp32):
//   cols [0,128) S buffer 0, [128,256) S buffer 1, [256,256+D) O accumulator.
// Shared memory (1024-byte aligned, all operands 128-byte swizzled):
//   Q tile, STAGES x K tile, STAGES x V tile, P tile (bf16), barriers.
// Per key tile j the MMA warp issues S_{j+1} = Q K_{j+1}^T before O += P_j V_j,
// so the tensor core computes the next scores while the softmax warps work
// on the current ones.
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int BR = kFwdBlockRows;
constexpr int BC = kFwdBlockCols;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kTmemO = 256;
// Lazy rescaling: the reference maximum of a row is raised only when a new
// score exceeds it by more than 2^8 in linear terms.  The final O / l uses
// the same reference for numerator and denominator, so the result is the
// same exact quantity; P stays <= 256 (bf16 and fp32 hold that easily).
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Cfg {
  static constexpr int STAGES = (D == 128) ? 2 : 3;
  static constexpr int BOXES = D / 64;         // 64-column (128-byte) boxes per row
  static constexpr int Q_BYTES = BR * D * 2;
  static constexpr int KV_BYTES = BC * D * 2;  // one K or one V tile
  static constexpr int P_BYTES = BR * BC * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], s_free[2], p_full, pv_done, drain
  static constexpr int NBAR = 1 + 3 * STAGES + 2 + 2 + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (u32) + abort flag (int)
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(kTmemO + D <= kTmemCols, "tensor memory budget");
};

struct Bars {
  uint32_t q_full, k_full0, v_full0, kv_empty0, s_full0, s_free0, p_full, pv_done, drain;
  __device__ uint32_t k_full(int s) const { return k_full0 + 8 * s; }
  __device__ uint32_t v_full(int s) const { return v_full0 + 8 * s; }
  __device__ uint32_t kv_empty(int s) const { return kv_empty0 + 8 * s; }
  __device__ uint32_t s_full(int b) const { return s_full0 + 8 * b; }
  __device__ uint32_t s_free(int b) const { return s_free0 + 8 * b; }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_bf16_sm103_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V, sP = sb + C::OFF_P;

  Bars bar;
  {
    uint32_t b = sb + C::OFF_BAR;
    bar.q_full = b;
    b += 8;
    bar.k_full0 = b;
    b += 8 * C::STAGES;
    bar.v_full0 = b;
    b += 8 * C::STAGES;
    bar.kv_empty0 = b;
    b += 8 * C::STAGES;
    bar.s_full0 = b;
    b += 16;
    bar.s_free0 = b;
    b += 16;
    bar.p_full = b;
    b += 8;
    bar.pv_done = b;
    b += 8;
    bar.drain = b;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqt = (p.N + BR - 1) / BR;
  const int bh = blockIdx.x / nqt;
  const int i0 = (blockIdx.x % nqt) * BR;
  const int N = p.N;
  const int r = p.window_r;

  // key tiles this query tile needs (only in-band tiles when windowed)
  int j_lo = 0, j_hi = (N + BC - 1) / BC;
  if (r >= 0) {
    const int lo = max(0, i0 - r);
    const int hi = min(N, i0 + BR + r);  // exclusive
    j_lo = lo / BC;
    j_hi = (hi + BC - 1) / BC;
  }
  const int ntiles = j_hi - j_lo;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.s_full(b), 1);
      mbar_init(bar.s_free(b), 4);  // one arrive per softmax warp
    }
    mbar_init(bar.p_full, 4);
    mbar_init(bar.pv_done, 1);
    mbar_init(bar.drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      prefetch_tensormap(&tmq);
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      mbar_arrive_expect_tx(bar.q_full, C::Q_BYTES);
#pragma unroll
      for (int b = 0; b < C::BOXES; ++b) tma_load_3d(sQ + b * BR * 128, &tmq, bar.q_full, b * 64, i0, bh);
      int issued = 0;
      for (int it = 0; it < ntiles; ++it) {
        const int st = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(bar.kv_empty(st), ph ^ 1, wc)) break;
        const int kv0 = (j_lo + it) * BC;
        mbar_arrive_expect_tx(bar.k_full(st), C::KV_BYTES);
#pragma unroll
        for (int b = 0; b < C::BOXES; ++b)
          tma_load_3d(sK + st * C::KV_BYTES + b * BC * 128, &tmk, bar.k_full(st), b * 64, kv0, bh);
        mbar_arrive_expect_tx(bar.v_full(st), C::KV_BYTES);
#pragma unroll
        for (int b = 0; b < C::BOXES; ++b)
          tma_load_3d(sV + st * C::KV_BYTES + b * BC * 128, &tmv, bar.v_full(st), b * 64, kv0, bh);
        issued = it + 1;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory is released
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.q_full, 0, drain);
        for (int it = max(0, issued - C::STAGES); it < issued; ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          mbar_wait(bar.k_full(st), ph, drain);
          mbar_wait(bar.v_full(st), ph, drain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BR, BC, 0, 0);  // Q: K-major, K tile: K-major
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BR, D, 0, 1);   // P: K-major, V tile: MN-major
      bool ok = mbar_wait(bar.q_full, 0, wc);
      auto issue_qk = [&](int it) -> bool {
        const int st = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        const int b = it & 1;
        if (!mbar_wait(bar.k_full(st), ph, wc)) return false;
        if (!mbar_wait(bar.s_free(b), ((it >> 1) & 1) ^ 1, wc)) return false;
        tc_fence_after();
        const uint32_t kbase = sK + st * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (BR * 128) + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * (BC * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + b * BC, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kbase + offk, 16, 1024),
                      idesc_qk, kk > 0);
        }
        mma_commit(bar.s_full(b));
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int it = 0; ok && it < ntiles; ++it) {
        if (it + 1 < ntiles && !issue_qk(it + 1)) break;
        const int st = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(bar.v_full(st), ph, wc)) break;
        if (!mbar_wait(bar.p_full, it & 1, wc)) break;
        tc_fence_after();
        const uint32_t vbase = sV + st * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk) {
          const uint32_t offp = (kk >> 2) * (BR * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + kTmemO, sdesc_sw128(sP + offp, 16, 1024),
                      sdesc_sw128(vbase + kk * 16 * 128, BC * 128, 1024), idesc_pv, (it > 0 || kk > 0));
        }
        mma_commit(bar.kv_empty(st));
        mma_commit(bar.pv_done);
      }
      // every MMA this thread issued must finish before tensor memory is freed
      mma_commit(bar.drain);
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(bar.drain, 0, drain);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const int qi = i0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl = p.scale_log2;
    float m_ref = -INFINITY;  // running reference maximum, log2 units of scaled scores
    float l = 0.f;
    bool ok = true;
    // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
    auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar_addr, parity, wc));
    };
    for (int it = 0; it < ntiles; ++it) {
      const int b = it & 1;
      if (!warp_wait(bar.s_full(b), (it >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[BC];
#pragma unroll
      for (int c = 0; c < BC / 32; ++c) tmem_ld_32x32b_x32(tl + b * BC + c * 32, &sr[c * 32]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.s_free(b));

      float s[BC];
#pragma unroll
      for (int c = 0; c < BC; ++c) s[c] = __uint_as_float(sr[c]);
      const int kv0 = (j_lo + it) * BC;
      const bool edge = (kv0 + BC > N) || (r >= 0 && !(kv0 >= i0 + BR - 1 - r && kv0 + BC - 1 <= i0 + r));
      if (edge) {
#pragma unroll
        for (int c = 0; c < BC; ++c) {
          const int kv = kv0 + c;
          const bool valid = kv < N && (r < 0 || abs(qi - kv) <= r);
          if (!valid) s[c] = -INFINITY;
        }
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < BC; ++c) mx = fmaxf(mx, s[c]);
      const float mt = mx * sl;
      float alpha = 1.f;
      if (mt > m_ref + kRescaleThreshold) {
        alpha = ex2_approx(m_ref - mt);  // 0 when m_ref = -inf
        m_ref = mt;
      }
      const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;
      float rs = 0.f;
      uint32_t pk[BC / 2];
#pragma unroll
      for (int c = 0; c < BC / 2; ++c) {
        const float p0 = ex2_approx(fmaf(s[2 * c], sl, -mref));
        const float p1 = ex2_approx(fmaf(s[2 * c + 1], sl, -mref));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;

      // P buffer and O accumulator are free once the previous P V has completed
      if (it > 0) {
        if (!warp_wait(bar.pv_done, (it - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tl + kTmemO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32x32b_x32(tl + kTmemO + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      // P row -> shared memory, K-major 128-byte swizzled (same layout TMA gives Q)
#pragma unroll
      for (int c16 = 0; c16 < BC / 8; ++c16) {
        const uint32_t addr = sP + (c16 >> 3) * (BR * 128) + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
        st_shared_v4(addr, pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full);
    }

    // ------------------------------------------------------------ epilogue
    const bool have = ok && warp_wait(bar.pv_done, (ntiles - 1) & 1);
    if (have) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      // stage the bf16 O tile in the (now idle) P buffer, swizzled like P
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tl + kTmemO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c16 = c * 4 + q4;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2 * e]) * inv_l,
                               __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv_l);
          const uint32_t addr = sP + (c16 >> 3) * (BR * 128) + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
          st_shared_v4(addr, w[0], w[1], w[2], w[3]);
        }
      }
      if (p.lse != nullptr && qi < N) {
        const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;
        p.lse[static_cast<size_t>(bh) * N + qi] = (mref + __log2f(l)) * 0.69314718055994531f;
      }
    }
    tc_fence_before();
    named_bar_sync(1, 128);  // reached by all four softmax warps on every path
    if (have && !*abort_flag) {
      // coalesced 128-bit stores: consecutive threads write consecutive 16-byte chunks
      constexpr int CHUNKS = D / 8;
      uint8_t* obase = reinterpret_cast<uint8_t*>(p.o) + (static_cast<size_t>(bh) * N + i0) * D * 2;
      for (int idx = row; idx < BR * CHUNKS; idx += 128) {
        const int rr = idx / CHUNKS, c16 = idx % CHUNKS;
        if (i0 + rr < N) {
          const uint4 val = ld_shared_v4(sP + (c16 >> 3) * (BR * 128) + rr * 128 + (((c16 & 7) ^ (rr & 7)) << 4));
          st_global_v4(obase + static_cast<size_t>(rr) * D * 2 + c16 * 16, val);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  using C = Cfg<D>;
  static bool configured = false;  // attribute set once per process (one device per process in practice)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_bf16_sm103_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long nqt = (p.N + BR - 1) / BR;
  const long long grid = nqt * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_fwd_bf16_sm103_kernel<D><<<static_cast<unsigned>(grid), kThreads, C::SMEM_BYTES, s>>>(m.q, m.k, m.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16_tc(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  if (p.d == 128) return launch_d<128>(p, m, s);
  if (p.d == 64) return launch_d<64>(p, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
