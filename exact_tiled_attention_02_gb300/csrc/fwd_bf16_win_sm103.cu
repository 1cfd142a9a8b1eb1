// fwd_bf16_win_sm103.cu -- tiled exact attention forward with a local window,
// bf16 in / fp32 accumulate, head dimensions 64, 96 and 128, for GB300
// (sm_103a).
//
// The computation is the one of fwd_bf16_sm103.cu: "Flash attention and
// efficient attention -- Hinglish notes", "The Standard Attention Problem",
// one key/value tile at a time with the running maximum / running sum merge
// of "Derivation: Incremental Softmax" (Steps 1-3), restricted to the band of
// "Worked example Local Attention Window" (query i sees key j iff
// |i - j| <= r): only the key tiles that meet the band are loaded.
//
// With a narrow band a query tile meets few key tiles (three for r = 128),
// so a CTA that pairs two query tiles spends much of each item filling and
// draining its pipeline: measured, the first tile's softmax idled about half
// of every item.  Here each CTA holds one query tile at a time, and two
// persistent CTAs per SM walk the query tiles; the launcher uses this kernel
// for r <= 128 (at most three key tiles per query tile); wider bands keep the
// two-tile persistent kernel,
// whose two-stage K/V ring hides the loads of long key loops (measured at
// 1 x 32 x 16384: w = 65, d = 128: 0.162 against 0.167 ms; w = 257: d = 64
// 0.126 against 0.138, d = 96 0.139 against 0.143, d = 128 0.151 both;
// w = 1025, d = 128: 0.298 against 0.275).  Here a CTA holds one 128-row query tile, with one S buffer
// and single K and V buffers, so that it takes 256 tensor-memory columns and
// under 100 KB of shared memory; two CTAs share each SM, and one CTA's loads,
// softmax and output overlap the other's products.  Per key tile j:
//   S_j = Q K_j^T (tcgen05.mma into TMEM), the softmax turns S_j into P_j
//   (bf16, over S's first 64 columns), O += P_j V_j.
// K_{j+1} loads as soon as S_j has read K_j, V_{j+1} as soon as P_j V_j has
// read V_j.  The O rescale needs no wait of its own: S_j's completion
// (s_full) implies P_{j-1} V_{j-1}'s, issued before it.
//
// CTA = 192 threads:
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t)
//   warp  4    TMEM owner + tcgen05.mma issuer (one elected lane)
//   warp  5    TMA producer (one elected lane)
// Tensor memory (256 columns): [0,128) S / P, [128, 128 + DP) O.
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int BR = kFwdBlockRows;  // 128 query rows per CTA
constexpr int BC = kFwdBlockCols;  // 128 keys per K/V tile
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;
constexpr uint32_t kTmemO = 128;
constexpr int BOX_BYTES = 128 * 128;  // a [128 rows][64 columns] bf16 box, 128-byte swizzled
constexpr float kRescaleThreshold = 8.0f;  // lazy rescaling (log2 units), as in the other forward kernels

template <int D>
struct CfgW {
  static_assert(D == 64 || D == 96 || D == 128, "head dimensions of this kernel");
  // tiles are DP columns wide in shared memory (whole 128-byte swizzle atoms;
  // at D = 96 the TMA zero-fills columns 96..127, and P V runs with N = 128,
  // because a 128-byte-swizzled MN-major V operand comes in 64-column atoms)
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int BOXES = DP / 64;
  static constexpr int TILE = BOXES * BOX_BYTES;
  static constexpr int OFF_Q = 0, OFF_K = TILE, OFF_V = 2 * TILE;
  static constexpr int OFF_OST = 3 * TILE;  // per softmax warp: 32 rows x 64 bytes of O (2 KB)
  static constexpr int OFF_BAR = OFF_OST + 4 * 2048;
  // q_full, k_full, k_empty, v_full, v_empty, s_full, p_full, o_done, drain, q_empty
  static constexpr int NBAR = 10;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (u32) + abort flag (int)
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // at least 80 KB, so that no more than two CTAs share an SM: tensor memory
  // holds two CTAs' 256 columns
  static constexpr int SMEM_BYTES = SMEM_USED + 1024 > 80 * 1024 ? SMEM_USED + 1024 : 80 * 1024;
  static_assert(2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
  static_assert(kTmemO + DP <= kTmemCols, "tensor memory budget");
};

struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full() const { return base + 8; }
  __device__ uint32_t k_empty() const { return base + 16; }
  __device__ uint32_t v_full() const { return base + 24; }
  __device__ uint32_t v_empty() const { return base + 32; }
  __device__ uint32_t s_full() const { return base + 40; }
  __device__ uint32_t p_full() const { return base + 48; }
  __device__ uint32_t o_done() const { return base + 56; }
  __device__ uint32_t drain() const { return base + 64; }
  __device__ uint32_t q_empty() const { return base + 72; }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    fa_fwd_bf16_win_sm103_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                                 const __grid_constant__ CUtensorMap tmv, const FwdParams p, int n_tiles) {
  using C = CfgW<D>;
  constexpr int DP = C::DP, TILE = C::TILE;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + C::SMEM_USED > static_cast<uint32_t>(C::SMEM_BYTES)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V;
  const Bars bar{sb + C::OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, r = p.window_r;
  const int nqt = (N + BR - 1) / BR;
  // query tile t of the CTA's list: its head, first row, and the key tiles
  // that meet its band
  struct Tile {
    int bh, i0, j_lo, ntiles;
  };
  auto tile_of = [&](int t) {
    Tile w;
    w.bh = t / nqt;
    w.i0 = (t % nqt) * BR;
    w.j_lo = max(0, w.i0 - r) / BC;
    w.ntiles = (min(N, min(N, w.i0 + BR) + r) + BC - 1) / BC - w.j_lo;
    return w;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full(), 1);
    mbar_init(bar.k_full(), 1);
    mbar_init(bar.k_empty(), 1);
    mbar_init(bar.v_full(), 1);
    mbar_init(bar.v_empty(), 1);
    mbar_init(bar.s_full(), 1);
    mbar_init(bar.p_full(), 4);  // one arrive per softmax warp
    mbar_init(bar.o_done(), 1);
    mbar_init(bar.drain(), 1);
    mbar_init(bar.q_empty(), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 5) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      prefetch_tensormap(&tmq);
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      bool ok = true;
      int g = 0, nt = 0;   // key tiles and query tiles of this CTA's list reached
      int kq = 0, vq = 0;  // K and V loads issued
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++nt) {
        const Tile w = tile_of(t);
        // Q once the previous tile's last S has read the old one
        if (nt > 0 && !mbar_wait_backoff(bar.q_empty(), (nt - 1) & 1, wc)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar.q_full(), TILE);
        for (int b = 0; b < C::BOXES; ++b) tma_load_3d(sQ + b * BOX_BYTES, &tmq, bar.q_full(), b * 64, w.i0, w.bh);
        // consumption order S_0, P_0 V_0, S_1, P_1 V_1, ... (across tiles): K
        // loads once the previous S has read K, V once the previous P V has
        // read V
        for (int j = 0; ok && j < w.ntiles; ++j, ++g) {
          const int kv0 = (w.j_lo + j) * BC;
          if (g > 0 && !mbar_wait_backoff(bar.k_empty(), (g - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar.k_full(), TILE);
          for (int b = 0; b < C::BOXES; ++b) tma_load_3d(sK + b * BOX_BYTES, &tmk, bar.k_full(), b * 64, kv0, w.bh);
          ++kq;
          if (g > 0 && !mbar_wait_backoff(bar.v_empty(), (g - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar.v_full(), TILE);
          for (int b = 0; b < C::BOXES; ++b) tma_load_3d(sV + b * BOX_BYTES, &tmv, bar.v_full(), b * 64, kv0, w.bh);
          ++vq;
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory is released
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        if (nt > 0) mbar_wait(bar.q_full(), (nt - 1) & 1, drain);
        if (kq > 0) mbar_wait(bar.k_full(), (kq - 1) & 1, drain);
        if (vq > 0) mbar_wait(bar.v_full(), (vq - 1) & 1, drain);
      }
    }
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BR, BC, 0, 0);  // Q, K: K-major
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BR, DP, 0, 1);  // P (TMEM), V: MN-major
      bool ok = true;
      int g = 0, nt = 0;  // key tiles and query tiles consumed
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++nt) {
        const Tile w = tile_of(t);
        if (!mbar_wait(bar.q_full(), nt & 1, wc)) break;
        for (int j = 0; j < w.ntiles; ++j, ++g) {
          // S_j = Q K_j^T (over P_{j-1}, which P_{j-1} V_{j-1}, issued before, has read)
          if (!mbar_wait(bar.k_full(), g & 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
            mma_bf16_ss(tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), idesc_qk, kk > 0);
          }
          mma_commit(bar.k_empty());
          if (j + 1 == w.ntiles) mma_commit(bar.q_empty());  // the tile's last reader of Q
          mma_commit(bar.s_full());
          // O (+)= P_j V_j.  The first P of a tile also means the softmax warps
          // have read the previous tile's O out of tensor memory.
          if (!mbar_wait2(bar.p_full(), g & 1, bar.v_full(), g & 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BC / 16; ++kk)
            mma_bf16_ts(tmem + kTmemO, tmem + kk * 8, sdesc_sw128(sV + kk * 16 * 128, BOX_BYTES, 1024), idesc_pv,
                        (j > 0 || kk > 0));
          mma_commit(bar.v_empty());
          mma_commit(bar.o_done());
        }
      }
      // every MMA this thread issued must finish before tensor memory is freed
      mma_commit(bar.drain());
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(bar.drain(), 0, drain);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t tO = tl + kTmemO;
    const float sl = p.scale_log2;
    bool ok = true;
    auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar_addr, parity, wc));
    };
    int g = 0;  // key tiles processed (all of this CTA's tiles)
    for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
    const Tile w = tile_of(t);
    const int bh = w.bh, i0 = w.i0, j_lo = w.j_lo, ntiles = w.ntiles;
    const int qi = i0 + row;
    const int qlo = i0, qhi = i0 + BR - 1;
    float m_ref = -INFINITY;  // running reference maximum, log2 units of scaled scores
    float l = 0.f;            // row sum of the unrounded P (lse uses it)
    float lc = 0.f;           // bf16 rounding error of each tile's largest P (O's normaliser adds it)
    for (int j = 0; j < ntiles; ++j, ++g) {
      if (!warp_wait(bar.s_full(), g & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[BC];
#pragma unroll
      for (int c = 0; c < BC / 32; ++c) tmem_ld_32x32b_x32(tl + c * 32, &sr[c * 32]);
      tmem_wait_ld();
      float s[BC];
#pragma unroll
      for (int c = 0; c < BC; ++c) s[c] = __uint_as_float(sr[c]);
      const int kv0 = (j_lo + j) * BC;
      if (kv0 + BC > N || !(kv0 >= qhi - r && kv0 + BC - 1 <= qlo + r)) {
        // the visible keys of row qi form one contiguous column range [lo, hi)
        const int lo = max(0, qi - r - kv0), hi = min(min(BC, N - kv0), qi + r + 1 - kv0);
        const unsigned span = hi > lo ? static_cast<unsigned>(hi - lo) : 0u;
#pragma unroll
        for (int c = 0; c < BC; ++c) s[c] = (static_cast<unsigned>(c - lo) < span) ? s[c] : -INFINITY;
      }
      float mx[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) mx[a] = fmaxf(s[a], s[a + 4]);
#pragma unroll
      for (int c = 8; c < BC; c += 8)
#pragma unroll
        for (int a = 0; a < 4; ++a) mx[a] = fmax3(mx[a], s[c + a], s[c + 4 + a]);
      const float smax = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      const float mt = smax * sl;
      float alpha = 1.f;
      if (mt > m_ref + kRescaleThreshold) {
        alpha = ex2_approx(m_ref - mt);  // 0 when m_ref = -inf
        m_ref = mt;
      }
      const float nref = (m_ref == -INFINITY) ? 0.f : -m_ref;
      // The tile's largest P, computed exactly as its element is below.  P V
      // multiplies bf16-rounded P while the row sum adds the unrounded
      // values; where one key dominates a row, that key's rounding (up to
      // 2^-9 of O: with lazy rescaling its P is 2^x, x in [0, 8]) is the whole
      // mismatch, and adding it to O's normaliser cancels it.
      const float pmax = ex2_approx(fmaf(smax, sl, nref));
      lc = lc * alpha + (bf16_round(pmax) - pmax);
      const float2 sl2 = make_float2(sl, sl), nref2 = make_float2(nref, nref);
      float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // P (bf16 pairs) over the first 64 columns of S, in groups of 16
      // columns; S columns 32g..32g+31 were read above, before group g
      // overwrites columns 16g..16g+15
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int e = 32 * g + 2 * c;
          const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), sl2, nref2);
          const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          rs[c & 3] = __fadd2_rn(rs[c & 3], pv);
          pk[c] = pack_bf16x2(pv.x, pv.y);
        }
        tmem_st_32x32b_x16(tl + 16 * g, pk);
      }
      const float rsum = (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y) + (rs[2].x + rs[2].y) + (rs[3].x + rs[3].y);
      // S_j has completed, and with it P_{j-1} V_{j-1}; P_j V_j waits for p_full
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < DP / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
            o[e] = __float_as_uint(v.x);
            o[e + 1] = __float_as_uint(v.y);
          }
          tmem_st_32x32b_x32(tO + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full());
      l = l * alpha + rsum;
    }

    // ------------------------------------------------------------ epilogue
    // The last P V has completed once o_done's last phase has.  Each warp
    // writes its 32 rows of O 32 columns (64 bytes a row) at a time through a
    // 2 KB staging buffer of its own: every thread puts its row's 64 bytes
    // there (16-byte chunk q of row r at position q ^ (r / 2 % 4), so that a
    // chunk of the 32 rows covers all eight 16-byte bank groups of a 128-byte
    // span), then the warp stores whole
    // 64-byte row segments, 8 rows per instruction (from registers, one row
    // per thread, each instruction touched 32 rows in 16-byte pieces).
    const bool have = ok && ntiles > 0 && warp_wait(bar.o_done(), (g - 1) & 1);
    if (have) {
      tc_fence_after();
      const float inv_l = 1.f / (l + lc);
      const uint32_t ost = sb + C::OFF_OST + (warp & 3) * 2048;
      const int r32 = lane;  // this thread's row within the warp's 32
      const int rbase = i0 + (warp & 3) * 32;
      uint8_t* obase = reinterpret_cast<uint8_t*>(p.o) + (static_cast<size_t>(bh) * N + rbase) * D * 2;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + c * 32, o);
        tmem_wait_ld();
        __syncwarp();  // the previous chunk's stores have read the buffer
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(ost + r32 * 64 + ((q4 ^ ((r32 >> 1) & 3)) << 4),
                       pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l),
                       pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l),
                       pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l),
                       pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l));
        __syncwarp();
        if (!*abort_flag) {
#pragma unroll
          for (int piece = 0; piece < 4; ++piece) {
            const int idx = piece * 32 + lane;  // 128 pieces of 16 bytes: row idx / 4, chunk idx % 4
            const int rr = idx >> 2, q4 = idx & 3;
            if (rbase + rr < N)
              st_global_v4(obase + static_cast<size_t>(rr) * D * 2 + c * 64 + q4 * 16,
                           ld_shared_v4(ost + rr * 64 + ((q4 ^ ((rr >> 1) & 3)) << 4)));
          }
        }
      }
      if (p.lse != nullptr && qi < N) {
        const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;
        p.lse[static_cast<size_t>(bh) * N + qi] = (mref + __log2f(l)) * 0.69314718055994531f;
      }
    }
    }  // tiles
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  constexpr int SMEM_BYTES = CfgW<D>::SMEM_BYTES;
  static bool configured = false;  // attribute set once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_bf16_win_sm103_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long tiles = static_cast<long long>((p.N + BR - 1) / BR) * p.BH;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return cudaErrorInvalidDevice;
  // persistent: two CTAs per SM walk the query tiles
  const long long grid = tiles < 2LL * sms ? tiles : 2LL * sms;
  fa_fwd_bf16_win_sm103_kernel<D><<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, s>>>(
      m.q, m.k, m.v, p, static_cast<int>(tiles));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16_win(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  if (p.window_r < 0) return cudaErrorInvalidValue;
  if (p.d == 128) return launch_d<128>(p, m, s);
  if (p.d == 96) return launch_d<96>(p, m, s);
  if (p.d == 64) return launch_d<64>(p, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
