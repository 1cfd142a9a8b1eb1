// fwd_bf16_d256_sm103.cu -- tiled exact attention forward for head
// dimension 256, bf16 in / fp32 accumulate, for GB300 (sm_103a).
//
// The same computation as the d <= 128 kernel (fwd_bf16_sm103.cu): "Flash
// attention and efficient attention -- Hinglish notes", "The Standard
// Attention Problem", evaluated one key/value tile at a time with the running
// maximum / running sum merge of that page's "Derivation: Incremental
// Softmax" (Steps 1-3) and of "Compute attention one tile at a time"
// (TensorViz), step "tiles"; the optional window of "Worked example Local
// Attention Window" skips the key tiles wholly outside the band.
//
// What changes at d = 256 is the on-chip budget:
//   * tensor memory (512 columns): one 128-row query tile per CTA, its O
//     accumulator (256 columns) and two S buffers (128 columns each), so
//     Q K_{j+1}^T runs on the tensor core while the softmax warps turn S_j
//     into P_j (a second query tile's O would not fit);
//   * shared memory: Q takes 64 KB and one 128-key K or V tile another 64 KB,
//     so K and V stream through a ring of five 32 KB chunks, each holding
//     128 keys x 128 of the 256 dimensions, loaded in the order the tensor
//     core consumes them:
//         K_0, K_1, V_0, K_2, V_1, K_3, ..., K_{T-1}, V_{T-2}, V_{T-1}
//     (two chunks each).  Every chunk is released by a tcgen05.commit right
//     after the products that read it, so loads run up to five chunks ahead.
// MMA issue order: S_0, S_1, then per key tile j: O += P_j V_j (two N = 128
// halves of O, one per V chunk), S_{j+2} = Q K_{j+2}^T into the buffer P_j
// occupied (tcgen05.mma operations of one thread execute in order, so S_{j+2}
// overwrites P_j only after P_j V_j has read it).
//
// CTA = 192 threads:
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t)
//   warp  4    TMEM owner + tcgen05.mma issuer (one elected lane)
//   warp  5    TMA producer (one elected lane)
// Tensor memory: [0,128) S_even / P_even, [128,256) S_odd / P_odd, [256,512) O.
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

// Shared-memory descriptor split in its two 32-bit words: the start address
// (bits 0-13) lives in the low word, so advancing it within one chunk is a
// 32-bit add (the field cannot carry: every address is below 256 KB), one
// instruction fewer per operand than a 64-bit add on the MMA warp (measured:
// 1.2-1.8% faster).
struct Desc2 {
  uint32_t lo, hi;
};
__device__ __forceinline__ Desc2 desc2(uint64_t d) {
  return Desc2{static_cast<uint32_t>(d), static_cast<uint32_t>(d >> 32)};
}
__device__ __forceinline__ void mma_ss2(uint32_t d_tmem, Desc2 a, uint32_t a_off, Desc2 b, uint32_t b_off,
                                        uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\n.reg .b64 da, db;\n"
      "mov.b64 da, {%1, %2};\nmov.b64 db, {%3, %4};\n"
      "setp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}\n" ::"r"(d_tmem),
      "r"(a.lo + a_off), "r"(a.hi), "r"(b.lo + b_off), "r"(b.hi), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts2(uint32_t d_tmem, uint32_t a_tmem, Desc2 b, uint32_t b_off, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\n.reg .b64 db;\n"
      "mov.b64 db, {%2, %3};\n"
      "setp.ne.b32 p, %5, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b.lo + b_off), "r"(b.hi), "r"(idesc), "r"(acc)
      : "memory");
}

constexpr int BR = kFwdBlockRows;  // 128 query rows per CTA
constexpr int BC = kFwdBlockCols;  // 128 keys per K/V tile
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr int BOX_BYTES = 128 * 128;           // a [128 rows][64 columns] bf16 box, 128-byte swizzled
constexpr int CHUNK_BYTES = 2 * BOX_BYTES;     // 128 rows x 128 columns

// D = 256 is the one instantiated.  D = 128 also fits (a six-chunk ring); it
// was measured as the single-query-tile point of the d = 128 tile-shape sweep
// and lost to the two-tile kernel of fwd_bf16_sm103.cu by 8-12%.
template <int D>
struct Cfg1 {
  static constexpr int CH = D / 128;                 // chunks per K or V tile
  static constexpr int Q_BYTES = (D / 64) * BOX_BYTES;
  static constexpr int NCHUNK = D == 256 ? 5 : 6;    // ring depth
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NCHUNK * CHUNK_BYTES;
  // q_full, full[NCHUNK], empty[NCHUNK], s_full[2], p_full[2], o_done, drain
  static constexpr int NBAR = 1 + 2 * NCHUNK + 6;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (u32) + abort flag (int)
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};
// Lazy rescaling threshold (log2 units), as in the d <= 128 kernel.
constexpr float kRescaleThreshold = 8.0f;

template <int NCHUNK>
struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t full(int c) const { return base + 8 * (1 + c); }
  __device__ uint32_t empty(int c) const { return base + 8 * (1 + NCHUNK + c); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 2 * NCHUNK + b); }
  // P_j of buffer b = j % 2 is in tensor memory.  One barrier per buffer: the
  // softmax may finish P_{j+1} before the MMA warp has waited for P_j, but it
  // cannot finish P_{j+2} (that needs S_{j+2}, issued after P_j V_j)
  __device__ uint32_t p_full(int b) const { return base + 8 * (3 + 2 * NCHUNK + b); }
  __device__ uint32_t o_done() const { return base + 8 * (5 + 2 * NCHUNK); }
  __device__ uint32_t drain() const { return base + 8 * (6 + 2 * NCHUNK); }
};

template <int D, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_bf16_d256_sm103_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                                  const __grid_constant__ CUtensorMap tmv, const FwdParams p) {
  using C = Cfg1<D>;
  constexpr int NCHUNK = C::NCHUNK, Q_BYTES = C::Q_BYTES, SMEM_USED = C::SMEM_USED, SMEM_BYTES = C::SMEM_BYTES;
  constexpr int OFF_Q = C::OFF_Q, OFF_RING = C::OFF_RING, OFF_BAR = C::OFF_BAR, OFF_MISC = C::OFF_MISC;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + SMEM_USED > static_cast<uint32_t>(SMEM_BYTES)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sQ = sb + OFF_Q, sRing = sb + OFF_RING;
  const Bars<NCHUNK> bar{sb + OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N;
  const int r = WIN ? p.window_r : -1;
  const int nqt = (N + BR - 1) / BR;
  const int bh = blockIdx.x / nqt;
  const int i0 = (blockIdx.x % nqt) * BR;

  // key tiles this query tile needs (only in-band tiles when windowed)
  int j_lo = 0, j_hi = (N + BC - 1) / BC;
  if (WIN) {
    j_lo = max(0, i0 - r) / BC;
    j_hi = (min(N, min(N, i0 + BR) + r) + BC - 1) / BC;
  }
  const int ntiles = j_hi - j_lo;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full(), 1);
    for (int c = 0; c < NCHUNK; ++c) {
      mbar_init(bar.full(c), 1);
      mbar_init(bar.empty(c), 1);
    }
    mbar_init(bar.s_full(0), 1);
    mbar_init(bar.s_full(1), 1);
    mbar_init(bar.p_full(0), 4);  // one arrive per softmax warp
    mbar_init(bar.p_full(1), 4);
    mbar_init(bar.o_done(), 1);
    mbar_init(bar.drain(), 1);
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
      mbar_arrive_expect_tx(bar.q_full(), Q_BYTES);
      for (int b = 0; b < D / 64; ++b) tma_load_3d(sQ + b * BOX_BYTES, &tmq, bar.q_full(), b * 64, i0, bh);
      int seq = 0;  // chunks issued
      bool ok = true;
      // the chunks (dimensions 0-127, 128-255, ...) of K or V tile j
      auto load_unit = [&](int j, bool is_v) {
        const int kv0 = (j_lo + j) * BC;
        for (int half = 0; half < C::CH && ok; ++half, ++seq) {
          const int c = seq % NCHUNK;
          if (!mbar_wait_backoff(bar.empty(c), ((seq / NCHUNK) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar.full(c), CHUNK_BYTES);
          for (int b = 0; b < 2; ++b)
            tma_load_3d(sRing + c * CHUNK_BYTES + b * BOX_BYTES, is_v ? &tmv : &tmk, bar.full(c),
                        half * 128 + b * 64, kv0, bh);
        }
      };
      if (ntiles > 0) load_unit(0, false);
      if (ntiles > 1) load_unit(1, false);
      for (int j = 0; ok && j < ntiles; ++j) {
        load_unit(j, true);
        if (j + 2 < ntiles) load_unit(j + 2, false);
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory is released
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.q_full(), 0, drain);
        for (int s = max(0, seq - NCHUNK); s < seq; ++s) mbar_wait(bar.full(s % NCHUNK), (s / NCHUNK) & 1, drain);
      }
    }
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BR, BC, 0, 0);   // Q, K chunk: K-major
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BR, 128, 0, 1);  // P (TMEM), V chunk: MN-major, N = 128
      int seq = 0;  // chunks consumed
      auto wait_chunk = [&](int& c) -> bool {
        c = seq % NCHUNK;
        if (!mbar_wait(bar.full(c), (seq / NCHUNK) & 1, wc)) return false;
        tc_fence_after();
        return true;
      };
      auto issue_s = [&](int j) -> bool {  // S_j = Q K_j^T into buffer j % 2
        const uint32_t d_tm = tmem + 128 * (j & 1);
        for (int half = 0; half < C::CH; ++half, ++seq) {
          int c;
          if (!wait_chunk(c)) return false;
          // descriptors built once, advanced by their address field per K-step
          const uint64_t dq = sdesc_sw128(sQ, 16, 1024), dk = sdesc_sw128(sRing + c * CHUNK_BYTES, 16, 1024);
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {  // 16 dimensions per step; 8 steps per chunk
            const int kk = half * 8 + k8;
            const uint32_t offq = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
            const uint32_t offk = (k8 >> 2) * BOX_BYTES + (k8 & 3) * 32;
            mma_ss2(d_tm, desc2(dq), offq >> 4, desc2(dk), offk >> 4, idesc_qk, kk > 0);
          }
          mma_commit(bar.empty(c));
        }
        mma_commit(bar.s_full(j & 1));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {  // O (+)= P_j V_j, one V chunk per half of O
        if (!mbar_wait(bar.p_full(j & 1), (j >> 1) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t a_tm = tmem + 128 * (j & 1);
        for (int half = 0; half < C::CH; ++half, ++seq) {
          int c;
          if (!wait_chunk(c)) return false;
          const uint64_t dv = sdesc_sw128(sRing + c * CHUNK_BYTES, BOX_BYTES, 1024);
#pragma unroll
          for (int kk = 0; kk < BC / 16; ++kk)
            mma_ts2(tmem + kTmemO + 128 * half, a_tm + kk * 8, desc2(dv), (kk * 16 * 128) >> 4, idesc_pv,
                        (j > 0 || kk > 0));
          mma_commit(bar.empty(c));
        }
        mma_commit(bar.o_done());
        return true;
      };
      bool ok = mbar_wait(bar.q_full(), 0, wc);
      if (ok && ntiles > 0) ok = issue_s(0);
      if (ok && ntiles > 1) ok = issue_s(1);
      for (int j = 0; ok && j < ntiles; ++j) {
        ok = issue_pv(j);
        if (ok && j + 2 < ntiles) ok = issue_s(j + 2);
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
    const int qi = i0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t tO = tl + kTmemO;
    const float sl = p.scale_log2;
    const int qlo = i0, qhi = i0 + BR - 1;
    float m_ref = -INFINITY;  // running reference maximum, log2 units of scaled scores
    float l = 0.f;            // row sum of the unrounded P (lse uses it)
    float lc = 0.f;           // bf16 rounding error of each tile's largest P (O's normaliser adds it)
    bool ok = true;
    auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar_addr, parity, wc));
    };
    for (int j = 0; j < ntiles; ++j) {
      if (!warp_wait(bar.s_full(j & 1), (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tl + 128 * (j & 1);
      uint32_t sr[BC];
#pragma unroll
      for (int c = 0; c < BC / 32; ++c) tmem_ld_32x32b_x32(tS + c * 32, &sr[c * 32]);
      tmem_wait_ld();
      float s[BC];
#pragma unroll
      for (int c = 0; c < BC; ++c) s[c] = __uint_as_float(sr[c]);
      const int kv0 = (j_lo + j) * BC;
      const bool edge = (kv0 + BC > N) || (WIN && !(kv0 >= qhi - r && kv0 + BC - 1 <= qlo + r));
      if (edge) {
        // the visible keys of row qi form one contiguous column range [lo, hi)
        int lo = 0, hi = min(BC, N - kv0);
        if (WIN) {
          lo = max(lo, qi - r - kv0);
          hi = min(hi, qi + r + 1 - kv0);
        }
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
      // P (bf16 pairs) over the first 64 columns of the S buffer, in groups of
      // 16 columns; S columns 32g..32g+31 were read above, before group g
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
        tmem_st_32x32b_x16(tS + 16 * g, pk);
      }
      const float rsum = (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y) + (rs[2].x + rs[2].y) + (rs[3].x + rs[3].y);
      // O may be rescaled only once the previous P V into it has completed.
      // Here P_{j-2} V_{j-2} has completed (S_j was issued after it) and
      // P_j V_j has not been issued, so o_done is within one phase of the
      // one waited for.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!warp_wait(bar.o_done(), (j - 1) & 1)) {
          tmem_wait_st();
          ok = false;
          break;
        }
        tc_fence_after();
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {  // 64 columns per round trip
          uint32_t o[64];
          tmem_ld_32x32b_x32(tO + 64 * c, &o[0]);
          tmem_ld_32x32b_x32(tO + 64 * c + 32, &o[32]);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
            o[e] = __float_as_uint(v.x);
            o[e + 1] = __float_as_uint(v.y);
          }
          tmem_st_32x32b_x32(tO + 64 * c, &o[0]);
          tmem_st_32x32b_x32(tO + 64 * c + 32, &o[32]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full(j & 1));
      l = l * alpha + rsum;
    }

    // ------------------------------------------------------------ epilogue
    // Up to two P V products may still be running here (S_{T-1} was issued
    // before P_{T-2} V_{T-2}), so o_done's parity cannot tell the last one
    // apart; the drain commit, issued after every MMA, can.  Q is idle once it
    // has completed: stage the bf16 O tile there, swizzled like Q's TMA layout.
    const bool have = ok && ntiles > 0 && warp_wait(bar.drain(), 0);
    if (have) {
      tc_fence_after();
      const float inv_l = 1.f / (l + lc);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c16 = c * 4 + q4;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2 * e]) * inv_l,
                               __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv_l);
          const uint32_t addr = sQ + (c16 >> 3) * BOX_BYTES + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
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
      constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
      uint8_t* obase = reinterpret_cast<uint8_t*>(p.o) + (static_cast<size_t>(bh) * N + i0) * D * 2;
      for (int idx = row; idx < BR * CHUNKS; idx += 128) {
        const int rr = idx / CHUNKS, c16 = idx % CHUNKS;
        if (i0 + rr < N) {
          const uint4 val = ld_shared_v4(sQ + (c16 >> 3) * BOX_BYTES + rr * 128 + (((c16 & 7) ^ (rr & 7)) << 4));
          st_global_v4(obase + static_cast<size_t>(rr) * D * 2 + c16 * 16, val);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool WIN>
cudaError_t launch_win(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  constexpr int SMEM_BYTES = Cfg1<D>::SMEM_BYTES;
  static bool configured = false;  // attribute set once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_bf16_d256_sm103_kernel<D, WIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long grid = static_cast<long long>((p.N + BR - 1) / BR) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_fwd_bf16_d256_sm103_kernel<D, WIN><<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, s>>>(m.q, m.k, m.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16_d256(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  if (p.d == 256) return p.window_r >= 0 ? launch_win<256, true>(p, m, s) : launch_win<256, false>(p, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
