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
// end.  Score tiles live only in tensor memory; nothing of size N x N reaches
// device memory.
//
// Work item = two 128-row query tiles (Q0, Q1) of one (batch, head).  The
// kernel is persistent: one CTA per SM (at most) takes items c, c + G,
// c + 2G, ... (G = the grid), every barrier's phase counting across items, so
// one item's start-up (loading Q and its first K/V tiles) overlaps the
// previous item's last products and output:
//   * the K/V ring runs on across items;
//   * Q_t of the next item is loaded once the current item's last Q_t K^T has
//     completed (the MMA warp commits q_empty(t) right after issuing it);
//   * O is written from registers (16-byte stores, one row per thread), not
//     staged in the Q buffer, which by then holds the next item's Q.
// (Measured against one item per CTA: identical results bit for bit, 2.6% to
// 7% faster on long key loops, 24% on the window-257 workload.)
// 384 threads (512 for unmasked d = 128):
//   warps 0-3  softmax for Q0: thread t owns row t of Q0 (TMEM lane t)
//   warps 4-7  softmax for Q1: thread t owns row t of Q1 (TMEM lane t)
//   warp  8    TMEM owner + tcgen05.mma issuer (one elected lane); for
//              unmasked d = 64 only the Q K^T products
//   warp  9    TMA producer (one elected lane)
//   warp  10   (unmasked d = 64) issues the P V products
//   warps 10-11 otherwise idle (registers are granted per warpgroup of four
//              warps, so a ten-warp CTA costs as much as twelve; 168 per thread)
//   warps 12-15 (unmasked d = 128) rescale O when a row's reference maximum
//              moves, one warp per TMEM lane quarter (see corr_warps)
// Tensor memory (512 columns x 128 lanes, 32-bit):
//   [0,128) S0 (P0 as packed bf16 in its first 64 columns), [128,256) S1 / P1,
//   [256,256+DP) O0, [384,384+DP) O1 (DP = D rounded up to 64: see Cfg);
//   unmasked d = 64: three S / P buffers [0,384) taken in turn, O0 at 384,
//   O1 at 448 (see tri_s).
// Shared memory (1024-byte aligned, 128-byte swizzled): Q0, Q1, a ring of
// STAGES K/V tiles, barriers.
// The two query tiles ping-pong: while the softmax warps of one tile turn
// S into P, the tensor core runs the other tile's P V and Q K^T, so the
// exponentials of one tile overlap the matrix products of the other.
// The softmax is instruction-issue bound, so it uses packed f32x2 FMA / add
// (two scores per instruction), three-input max, and ex2 on the
// special-function unit for every score.  Per key
// tile j the MMA warp issues  O0 += P0 V_j,  S0 = Q0 K_{j+1}^T,  O1 += P1 V_j,
// S1 = Q1 K_{j+1}^T; tcgen05.mma operations issued by one thread execute in
// order, so S_i(j+1) overwrites the columns of P_i(j) only after P_i(j) V_j
// has read them.
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int BR = kFwdBlockRows;  // rows per query tile (two per item)
constexpr int BC = kFwdBlockCols;  // keys per K/V tile
// The unmasked d = 128 instantiation adds a fourth warpgroup (warps 12-15)
// that rescales O when a row's reference maximum moves, so that the softmax
// warps need not.  Measured on 2x16x8192x128 with Q,K x8 (frequent
// rescales): forward 0.758 -> 0.727 ms; with few rescales (standard-normal
// inputs) it cost 1.5% at d = 128 and 1.3-3.3% at d = 96 and 64, which keep
// the rescale in the softmax warps.
template <int D, bool WIN>
constexpr bool corr_warps() {
  return !WIN && D == 128;  // the alpha region in shared memory exists only at D = 128
}
template <int D, bool WIN>
constexpr int threads_for() {
  return corr_warps<D, WIN>() ? 512 : 384;
}
// register shares with the correction warpgroup (512 threads x 128 at
// launch): softmax warpgroups 152, the other two 104 (2 x 152 + 2 x 104 = 4 x 128)
constexpr int kRegsSoftmax = 152;
constexpr int kRegsOther = 104;
static_assert(2 * kRegsSoftmax + 2 * kRegsOther == 4 * 128, "register shares must add up to the launch allocation");
constexpr int kTmemCols = 512;
// Unmasked d = 64 keeps three S buffers instead of two: its S and O of both
// tiles take 2 x (128 + 64) columns, and the last 128 hold a third S, so that
// the S of a tile's next key tile is computed a whole step ahead, and it
// issues its products from two threads (S from warp 8, P V from warp 10).
// Measured on 4x16x2048x64: one S per tile and one issuing thread, 2665
// cycles per key step for 1280 cycles of products; three buffers, 2650
// (a single issuer spent ~1100 cycles a step on waits and bookkeeping between
// instructions, each of which takes about as long to issue as to execute at
// these sizes); three buffers and two issuers, ~2250; forward 0.0963 ->
// 0.0761 ms.
template <int D, bool WIN>
constexpr bool tri_s() {
  return D == 64 && !WIN;
}
constexpr uint32_t tm_s(int b) { return 128u * static_cast<uint32_t>(b); }  // S buffer b (P over its first half)
template <int D, bool WIN>
constexpr uint32_t tm_o(int t) {  // O of query tile t
  return tri_s<D, WIN>() ? 384u + 64u * static_cast<uint32_t>(t) : 256u + 128u * static_cast<uint32_t>(t);
}
// Lazy rescaling: a row's reference maximum is raised only when a new score
// exceeds it by more than 2^8 in linear terms.  The final O / l uses the same
// reference for numerator and denominator, so the result is the same exact
// quantity; P stays <= 256.  (Measured on the large-logit workload: larger
// thresholds save up to 3% of the time but raise the mean output error, from
// 3.7e-4 at 2^8 to 6.1e-4 at 2^64.)
constexpr float kRescaleThreshold = 8.0f;

// Shared-memory descriptor split in its two 32-bit words: the start address
// (bits 0-13) lives in the low word, so advancing it within one tile is a
// 32-bit add (the field cannot carry: every address is below 256 KB), one
// instruction fewer per operand than a 64-bit add on the MMA warp, which
// shares its SM sub-partition with two softmax warps.  Measured: 2.0-2.4%
// faster at d = 128, 1.2% at d = 96; at d = 64 the 64-bit form measured
// 2.4% faster, so that instantiation keeps it.
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

// D = 64, 96 or 128.  Tiles in shared memory are DP = D rounded up to a
// multiple of 64 columns wide (whole 128-byte swizzle atoms); for D = 96 the
// TMA zero-fills columns 96..127.  Q K^T contracts over the D real columns
// only.  P V runs with N = DP: a 128-byte-swizzled MN-major V operand is laid
// out in 64-column atoms, so N = 96 is not one of its layouts, and the zero
// columns of V only produce zero columns of O, which are never read.
template <int D>
struct Cfg {
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int STAGES = (DP == 128) ? 2 : 3;
  static constexpr int BOXES = DP / 64;
  static constexpr int Q_BYTES = BR * DP * 2;
  static constexpr int KV_BYTES = BC * DP * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  // q_full[2], q_empty[2], k_full[S], v_full[S], kv_empty[S], s_full[3], p_full[3], o_done[2], drain,
  // o_staged[2], o_free, alpha_ready[2], pv_done[3]
  static constexpr int NBAR = 4 + 3 * STAGES + 17;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // D = 64 leaves room for an output staging tile (bf16 [BR][DP]) that the
  // two query tiles share in turn; at DP = 128 the K/V ring takes that space
  static constexpr bool STAGED_OUT = (DP == 64);
  // each row's rescale factor, handed from the softmax to the correction
  // warps (d = 128 only; elsewhere the extra shared memory cost L1 and time)
  static constexpr int OFF_ALPHA = (OFF_MISC + 16 + 127) / 128 * 128;  // float [2][BR]
  static constexpr int OFF_OST = OFF_ALPHA + (D == 128 ? 2 * BR * 4 : 0);
  static constexpr int SMEM_USED = STAGED_OUT ? OFF_OST + BR * DP * 2 : OFF_OST;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(D % 32 == 0 && DP <= 128, "tensor memory budget");
};

template <int STAGES>
struct Bars {
  uint32_t base;
  __device__ uint32_t q_full(int t) const { return base + 8 * t; }
  __device__ uint32_t q_empty(int t) const { return base + 8 * (2 + t); }
  __device__ uint32_t k_full(int s) const { return base + 8 * (4 + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (4 + STAGES + s); }
  __device__ uint32_t kv_empty(int s) const { return base + 8 * (4 + 2 * STAGES + s); }
  // s_full / p_full: one per S buffer (the query tile's index where a tile owns its buffer)
  __device__ uint32_t s_full(int b) const { return base + 8 * (4 + 3 * STAGES + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (7 + 3 * STAGES + b); }
  __device__ uint32_t o_done(int t) const { return base + 8 * (10 + 3 * STAGES + t); }
  __device__ uint32_t drain() const { return base + 8 * (12 + 3 * STAGES); }
  __device__ uint32_t o_staged(int t) const { return base + 8 * (13 + 3 * STAGES + t); }
  __device__ uint32_t o_free() const { return base + 8 * (15 + 3 * STAGES); }
  __device__ uint32_t alpha_ready(int t) const { return base + 8 * (16 + 3 * STAGES + t); }
  // three-buffer layout: the P V that read S buffer b has completed
  __device__ uint32_t pv_done(int b) const { return base + 8 * (18 + 3 * STAGES + b); }
};

// The key tiles of one item: [j_lo, j_lo + ntiles), and each query tile's own
// range as offsets into it (only in-band tiles when windowed).
struct Item {
  int bh, i0, j_lo, ntiles;
  int lo[2], hi[2];
};

// Items [0, n_pair) are pairs of query tiles.  Unmasked, when the last round
// of pairs would fill at most half the CTAs, the launcher passes n_pair
// smaller than the number of pairs and the remaining pairs run as single
// query tiles, items n_pair, n_pair + 1, ... (item n_pair + s holds tile s % 2
// of pair n_pair + s / 2; its second tile is empty), so that they spread over
// twice as many CTAs.
template <bool WIN>
__device__ __forceinline__ Item decode_item(int item, int N, int r, int n_pair) {
  Item w;
  const int nqt = (N + 2 * BR - 1) / (2 * BR);
  if (!WIN && item >= n_pair) {
    const int s = item - n_pair, pair = n_pair + s / 2;
    w.bh = pair / nqt;
    w.i0 = (pair % nqt) * (2 * BR) + (s & 1) * BR;
    w.j_lo = 0;
    // a tile wholly past N (the second tile of a head's last pair) makes an
    // empty item: no key tiles, so no role loads or waits for any
    w.ntiles = w.i0 < N ? (N + BC - 1) / BC : 0;
    w.lo[0] = 0;
    w.hi[0] = w.ntiles;
    w.lo[1] = 0;
    w.hi[1] = 0;
    return w;
  }
  w.bh = item / nqt;
  w.i0 = (item % nqt) * (2 * BR);
  w.j_lo = 0;
  int j_hi = (N + BC - 1) / BC;
  if (WIN) {
    w.j_lo = max(0, w.i0 - r) / BC;
    j_hi = (min(N, w.i0 + 2 * BR + r) + BC - 1) / BC;
  }
  w.ntiles = j_hi - w.j_lo;
  for (int t = 0; t < 2; ++t) {
    w.lo[t] = 0;
    w.hi[t] = w.ntiles;
    const int row_lo = w.i0 + t * BR, row_hi = min(N, row_lo + BR) - 1;
    if (WIN) {
      if (row_lo >= N) {
        w.hi[t] = 0;
      } else {
        w.lo[t] = max(0, row_lo - r) / BC - w.j_lo;
        w.hi[t] = (min(N, row_hi + r + 1) + BC - 1) / BC - w.j_lo;
      }
    }
  }
  return w;
}

template <int D, bool WIN>
__global__ void __launch_bounds__(threads_for<D, WIN>(), 1)
    fa_fwd_bf16_sm103_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                                     const __grid_constant__ CUtensorMap tmv, const FwdParams p, int n_items,
                                     int n_pair) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + C::SMEM_USED > static_cast<uint32_t>(C::SMEM_BYTES)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V, sOst = sb + C::OFF_OST;
  const Bars<C::STAGES> bar{sb + C::OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N;
  const int r = WIN ? p.window_r : -1;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar.q_full(t), 1);
      mbar_init(bar.q_empty(t), 1);
      mbar_init(bar.alpha_ready(t), 4);
      mbar_init(bar.o_done(t), 1);
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(bar.s_full(b), 1);
      mbar_init(bar.p_full(b), corr_warps<D, WIN>() ? 8 : 4);  // the softmax warps of a tile (+ correction warps)
      mbar_init(bar.pv_done(b), 1);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.v_full(s), 1);
      // three-buffer layout: released by both MMA issuers (the S and the P V products)
      mbar_init(bar.kv_empty(s), tri_s<D, WIN>() ? 2 : 1);
    }
    mbar_init(bar.drain(), tri_s<D, WIN>() ? 2 : 1);
    mbar_init(bar.o_staged(0), 128);  // staged output: every thread of the tile, after its row
    mbar_init(bar.o_staged(1), 128);
    mbar_init(bar.o_free(), 4);       // ... one arrive per warp of the tile that just stored
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The roles, one lambda each.  Unmasked d = 128 adds the correction warps
  // and moves registers between warpgroups (one setmaxnreg instruction per
  // warpgroup, at the top of its branch); the other instantiations keep the
  // twelve-warp layout, whose code measured faster there.
  auto role_correction = [&]() {
    // ------------------------------------------------------------ correction
    // (unmasked d = 128) Warp 12 + q rescales the O rows in TMEM lane
    // quarter q of both query tiles when a row's reference maximum has
    // moved: after the tile's previous P V into O has completed and before
    // its next one (p_full counts these warps too), while the softmax warps
    // go on computing P.
    if constexpr (corr_warps<D, WIN>()) {
      const int q = warp & 3;
      const uint32_t tlq = tmem + (static_cast<uint32_t>(q * 32) << 16);
      const float* sAlpha = reinterpret_cast<const float*>(smem + C::OFF_ALPHA);
      auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar_addr, parity, wc));
      };
      int nt[2] = {0, 0};  // key tiles each query tile has passed (all items)
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const Item w = decode_item<WIN>(item, N, r, n_pair);
        for (int it = 0; ok && it < w.ntiles; ++it) {
          for (int t = 0; t < 2; ++t) {
            if (it < w.lo[t] || it >= w.hi[t]) continue;
            if (!warp_wait(bar.alpha_ready(t), nt[t] & 1)) {
              ok = false;
              break;
            }
            const float a = sAlpha[t * BR + q * 32 + lane];
            if (it > w.lo[t] && __any_sync(0xffffffffu, a != 1.f)) {
              if (!warp_wait(bar.o_done(t), (nt[t] - 1) & 1)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t tO = tlq + tm_o<D, WIN>(t);
              const float2 a2 = make_float2(a, a);
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(tO + c * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
                  o[e] = __float_as_uint(v.x);
                  o[e + 1] = __float_as_uint(v.y);
                }
                tmem_st_32x32b_x32(tO + c * 32, o);
              }
              tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar.p_full(t));
            ++nt[t];
          }
        }
      }
    }
  };
  auto role_tma = [&]() {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      prefetch_tensormap(&tmq);
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      bool ok = true;
      int g = 0;         // ring slots issued so far (all items)
      int nq = 0;        // items whose Q was issued
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++nq) {
        const Item w = decode_item<WIN>(item, N, r, n_pair);
        for (int t = 0; t < 2; ++t) {
          // the previous item's last Q_t K^T has completed
          if (nq > 0 && !mbar_wait_backoff(bar.q_empty(t), (nq - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar.q_full(t), C::Q_BYTES);
#pragma unroll
          for (int b = 0; b < C::BOXES; ++b)
            tma_load_3d(sQ + t * C::Q_BYTES + b * BR * 128, &tmq, bar.q_full(t), b * 64, w.i0 + t * BR, w.bh);
        }
        for (int it = 0; ok && it < w.ntiles; ++it, ++g) {
          const int st = g % C::STAGES;
          if (!mbar_wait_backoff(bar.kv_empty(st), ((g / C::STAGES) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          const int kv0 = (w.j_lo + it) * BC;
          // three-buffer layout: K and V of a slot complete one barrier, so a
          // P (computed from an S that read K) implies its V is resident too
          const uint32_t vbar = tri_s<D, WIN>() ? bar.k_full(st) : bar.v_full(st);
          mbar_arrive_expect_tx(bar.k_full(st), tri_s<D, WIN>() ? 2 * C::KV_BYTES : C::KV_BYTES);
#pragma unroll
          for (int b = 0; b < C::BOXES; ++b)
            tma_load_3d(sK + st * C::KV_BYTES + b * BC * 128, &tmk, bar.k_full(st), b * 64, kv0, w.bh);
          if (!tri_s<D, WIN>()) mbar_arrive_expect_tx(bar.v_full(st), C::KV_BYTES);
#pragma unroll
          for (int b = 0; b < C::BOXES; ++b)
            tma_load_3d(sV + st * C::KV_BYTES + b * BC * 128, &tmv, vbar, b * 64, kv0, w.bh);
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory is released
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        if (nq > 0) {
          mbar_wait(bar.q_full(0), (nq - 1) & 1, drain);
          mbar_wait(bar.q_full(1), (nq - 1) & 1, drain);
        }
        for (int s = max(0, g - C::STAGES); s < g; ++s) {
          mbar_wait(bar.k_full(s % C::STAGES), (s / C::STAGES) & 1, drain);
          if (!tri_s<D, WIN>()) mbar_wait(bar.v_full(s % C::STAGES), (s / C::STAGES) & 1, drain);
        }
      }
    }
    __syncwarp();
  };
  auto role_mma = [&]() {
    // ------------------------------------------------------------------ MMA (warp 8)
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BR, BC, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BR, C::DP, 0, 1);
      int g0 = 0;               // ring slot of the current item's first key tile
      int cnt[2] = {0, 0};      // key tiles each query tile has processed (all items)
      int nq = 0;               // items started
      int last[2] = {0, 0};     // index of each tile's last key tile in the current item
      // three-buffer layout: S products issued (all items), the buffer of the
      // next one and that buffer's phase parity; the K/V ring slot and parity
      int ks = 0, bs = 0, rs = 0;
      uint32_t bq = 0, rp = 0;
      auto issue_s = [&](int t, int it, int b) {  // S_t = Q_t K_it^T into S buffer b
        // descriptors built once per tile, advanced by their address field
        // (16-byte units) per K-step: the MMA warp shares its SM
        // sub-partition with two softmax warps, and rebuilding both 64-bit
        // descriptors for every instruction made issuing slower than the
        // tensor core (measured: 3-4% on long key loops).  Every sum is
        // still a shared-memory address below 256 KB, so the 14-bit field
        // never carries into the neighbouring offset fields.
        const uint64_t dq = sdesc_sw128(sQ + t * C::Q_BYTES, 16, 1024);
        const uint64_t dk = sdesc_sw128(sK + ((g0 + it) % C::STAGES) * C::KV_BYTES, 16, 1024);
        const uint32_t dt = tmem + tm_s(b);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offq = (kk >> 2) * (BR * 128) + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * (BC * 128) + (kk & 3) * 32;
          if constexpr (D != 64)
            mma_ss2(dt, desc2(dq), offq >> 4, desc2(dk), offk >> 4, idesc_qk, kk > 0);
          else
            mma_bf16_ss(dt, dq + (offq >> 4), dk + (offk >> 4), idesc_qk, kk > 0);
        }
        mma_commit(bar.s_full(b));
        if (it == last[t]) mma_commit(bar.q_empty(t));  // Q_t is free once this product completes
      };
      auto issue_pv = [&](int t, int it, bool first, int b) {  // O_t (+)= P_t V_it, P_t in S buffer b
        const uint64_t dv = sdesc_sw128(sV + ((g0 + it) % C::STAGES) * C::KV_BYTES, BC * 128, 1024);
        const uint32_t dt = tmem + tm_o<D, WIN>(t), at = tmem + tm_s(b);
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk)
          if constexpr (D != 64)
            mma_ts2(dt, at + kk * 8, desc2(dv), (kk * 16 * 128) >> 4, idesc_pv, (!first || kk > 0));
          else
            mma_bf16_ts(dt, at + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc_pv, (!first || kk > 0));
        mma_commit(bar.o_done(t));
      };
      auto wait_k = [&](int it) {
        const int g = g0 + it;
        return mbar_wait(bar.k_full(g % C::STAGES), (g / C::STAGES) & 1, wc);
      };
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++nq) {
        const Item w = decode_item<WIN>(item, N, r, n_pair);
        ok = mbar_wait2(bar.q_full(0), nq & 1, bar.q_full(1), nq & 1, wc);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          last[t] = w.hi[t] - 1;
          if (w.lo[t] >= w.hi[t]) mma_commit(bar.q_empty(t));  // no product reads Q_t in this item
        }
        if constexpr (tri_s<D, WIN>()) {
          // Three S buffers, taken in turn by the S products in issue order
          // (index ks counts them across items): S0(0) S1(0) S0(1) S1(1) ...
          // for a pair of tiles, S(0) S(1) ... for a single tile.  This
          // thread issues only the S products; warp 10 issues the P V
          // products (role_pv), so that neither thread's waits and
          // bookkeeping hold up the tensor core (one thread issuing every
          // product left it idle about half the time: issuing an
          // instruction takes nearly as long as executing one at these
          // sizes).  S(k) overwrites buffer k % 3 once the P V that read
          // S(k - 3) there has completed (pv_done), so every tile's next S
          // is computed while its softmax works on the current one.
          const bool pair = w.lo[1] < w.hi[1];
          for (int it = 0; ok && it < w.ntiles; ++it) {
            if (!mbar_wait(bar.k_full(rs), rp, wc)) {  // K_it and V_it resident
              ok = false;
              break;
            }
            for (int t = 0; t < (pair ? 2 : 1); ++t) {
              if (ks >= 3 && !mbar_wait(bar.pv_done(bs), bq ^ 1u, wc)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(t, it, bs);
              ++ks;
              if (++bs == 3) {
                bs = 0;
                bq ^= 1u;
              }
            }
            if (!ok) break;
            mma_commit(bar.kv_empty(rs));  // this issuer's share of the slot's release
            if (++rs == C::STAGES) {
              rs = 0;
              rp ^= 1u;
            }
          }
        } else if (!WIN && w.lo[1] < w.hi[1]) {
          // both tiles take every key tile: PV0(j), S0(j+1), PV1(j), release, S1(j+1)
          ok = wait_k(0);
          if (ok) {
            tc_fence_after();
            issue_s(0, 0, 0);
            issue_s(1, 0, 1);
          }
          for (int it = 0; ok && it < w.ntiles; ++it) {
            const int g = g0 + it;
            const int st = g % C::STAGES;
            const bool more = it + 1 < w.ntiles;
            // V_j and P0_j in one round trip (see mbar_wait2); with a three-deep
            // ring the next K is resident by then too (measured: +3% at d = 64),
            // with two it may still be in flight (-5% at d = 128 when waited
            // for here), so it gets its own wait after P0 V_j
            const uint32_t pv = (g / C::STAGES) & 1, pp = (cnt[0] + it) & 1;
            constexpr bool k_early = C::STAGES >= 3;
            if (k_early && more ? !mbar_wait3(bar.v_full(st), pv, bar.p_full(0), pp, bar.k_full((g + 1) % C::STAGES),
                                              ((g + 1) / C::STAGES) & 1, wc)
                                : !mbar_wait2(bar.v_full(st), pv, bar.p_full(0), pp, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(0, it, it == 0, 0);
            if (more) {
              if (!k_early) {
                if (!wait_k(it + 1)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              issue_s(0, it + 1, 0);
            }
            if (!mbar_wait(bar.p_full(1), (cnt[1] + it) & 1, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(1, it, it == 0, 1);
            mma_commit(bar.kv_empty(st));  // before S1(j+1): a commit waits for every earlier MMA
            if (more) issue_s(1, it + 1, 1);
          }
          cnt[0] += w.ntiles;
          cnt[1] += w.ntiles;
        } else {
          // windowed, or a single-tile item: each tile only over its own key range
          for (int t = 0; t < 2; ++t) {
            if (!ok || w.lo[t] >= w.hi[t]) continue;
            ok = wait_k(w.lo[t]);
            if (ok) {
              tc_fence_after();
              issue_s(t, w.lo[t], t);
            }
          }
          int c[2] = {0, 0};
          for (int it = 0; ok && it < w.ntiles; ++it) {
            const int g = g0 + it;
            const int st = g % C::STAGES;
            if (!mbar_wait(bar.v_full(st), (g / C::STAGES) & 1, wc)) {
              ok = false;
              break;
            }
            bool k_next = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!ok || it < w.lo[t] || it >= w.hi[t]) continue;
              if (!mbar_wait(bar.p_full(t), (cnt[t] + c[t]) & 1, wc)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_pv(t, it, c[t] == 0, t);
              ++c[t];
              if (t == 1 || it < w.lo[1] || it >= w.hi[1]) mma_commit(bar.kv_empty(st));
              if (it + 1 < w.hi[t]) {
                if (!k_next && !(k_next = wait_k(it + 1))) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                issue_s(t, it + 1, t);
              }
            }
          }
          cnt[0] += c[0];
          cnt[1] += c[1];
        }
        g0 += w.ntiles;
      }
      // every MMA this thread issued must finish before tensor memory is freed
      mma_commit(bar.drain());
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(bar.drain(), 0, drain);
    }
    __syncwarp();
  };
  auto role_pv = [&]() {
    // ---------------------------------------------- P V issuer (warp 10)
    // (three-buffer layout) O_t += P_t V_j for every P in the order the S
    // products were issued: the k-th P lives in S buffer k % 3 and completes
    // phase k / 3 of that buffer's p_full barrier.  A P implies its V is
    // resident: K and V of a slot complete one barrier, which the S product
    // that P was computed from waited for.
    if constexpr (tri_s<D, WIN>()) {
      if (lane == 0) {
        constexpr uint32_t idesc_pv = idesc_bf16_f32(BR, C::DP, 0, 1);
        int bs = 0, rs = 0;
        uint32_t bq = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
          const Item w = decode_item<WIN>(item, N, r, n_pair);
          const bool pair = w.lo[1] < w.hi[1];
          for (int it = 0; ok && it < w.ntiles; ++it) {
            const uint64_t dv = sdesc_sw128(sV + rs * C::KV_BYTES, BC * 128, 1024);
            for (int t = 0; t < (pair ? 2 : 1); ++t) {
              if (!mbar_wait(bar.p_full(bs), bq, wc)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t dt = tmem + tm_o<D, WIN>(t), at = tmem + tm_s(bs);
#pragma unroll
              for (int kk = 0; kk < BC / 16; ++kk)
                mma_bf16_ts(dt, at + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc_pv, (it > 0 || kk > 0));
              mma_commit(bar.o_done(t));
              mma_commit(bar.pv_done(bs));
              if (++bs == 3) {
                bs = 0;
                bq ^= 1u;
              }
            }
            if (!ok) break;
            mma_commit(bar.kv_empty(rs));  // this issuer's share of the slot's release
            if (++rs == C::STAGES) rs = 0;
          }
        }
        // every product this thread issued must finish before tensor memory is freed
        mma_commit(bar.drain());
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.drain(), 0, drain);
      }
      __syncwarp();
    }
  };
  auto role_softmax = [&]() {
    // -------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tO = tl + tm_o<D, WIN>(t);
    const float sl = p.scale_log2;
    bool ok = true;
    // windowed items are short, and there the staged path measured 7% slower
    constexpr bool kStagedOut = C::STAGED_OUT && !WIN;
    int n = 0;   // key tiles this warpgroup has processed (all items)
    int ni = 0;  // items this warpgroup has passed (both warpgroups see every item)
    int no = 0;  // outputs this warpgroup has staged
    int ks = 0;  // S products of all items before this one (three-buffer layout; as counted by the MMA role)
    auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar_addr, parity, wc));
    };
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const Item w = decode_item<WIN>(item, N, r, n_pair);
      const int qi = w.i0 + t * BR + row;
      const int qlo = w.i0 + t * BR, qhi = qlo + BR - 1;
      // l: row sum of the unrounded P (lse uses it); lc: the bf16 rounding
      // error of each tile's largest P, which O's normaliser adds (below)
      float m_ref = -INFINITY, l = 0.f, lc = 0.f;
      const bool pair = w.lo[1] < w.hi[1];
      for (int it = w.lo[t]; it < w.hi[t]; ++it, ++n) {
        // this tile's S buffer and the phase it completes there
        int sb = t;
        uint32_t sph = n & 1;
        int k = 0;  // (three-buffer layout) index of this S product among all issued
        if constexpr (tri_s<D, WIN>()) {
          k = pair ? ks + 2 * it + t : ks + it;
          sb = k % 3;
          sph = (k / 3) & 1;
        }
        const uint32_t tS = tl + tm_s(sb);
        if (!warp_wait(bar.s_full(sb), sph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[BC];
#pragma unroll
        for (int c = 0; c < BC / 32; ++c) tmem_ld_32x32b_x32(tS + c * 32, &sr[c * 32]);
        tmem_wait_ld();
        float s[BC];
#pragma unroll
        for (int c = 0; c < BC; ++c) s[c] = __uint_as_float(sr[c]);
        const int kv0 = (w.j_lo + it) * BC;
        const bool edge = (kv0 + BC > N) || (WIN && !(kv0 >= qhi - r && kv0 + BC - 1 <= qlo + r));
        if (edge) {
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
          alpha = ex2_approx(m_ref - mt);
          m_ref = mt;
        }
        if constexpr (corr_warps<D, WIN>()) {
          // the correction warp of this lane quarter rescales O meanwhile
          reinterpret_cast<float*>(smem + C::OFF_ALPHA)[t * BR + row] = alpha;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar.alpha_ready(t));
        }
        const float nref = (m_ref == -INFINITY) ? 0.f : -m_ref;
        // The tile's largest P, computed exactly as its element is below
        // (same fused multiply-add, same exp2).  P V multiplies the bf16
        // rounding of every P, and the row sum adds the unrounded values; in
        // a row that one key dominates (large logits) that mismatch is the
        // dominant key's rounding, up to 2^-9 of O, because with lazy
        // rescaling that P is 2^x, x in [0, 8], not exactly 1.  Adding the
        // largest P's rounding error to O's normaliser cancels it.
        const float pmax = ex2_approx(fmaf(smax, sl, nref));
        lc = lc * alpha + (bf16_round(pmax) - pmax);
        const float2 sl2 = make_float2(sl, sl), nref2 = make_float2(nref, nref);
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int gq = 0; gq < BC / 32; ++gq) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int e = 32 * gq + 2 * c;
            const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), sl2, nref2);
            const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            rs[c & 3] = __fadd2_rn(rs[c & 3], pv);
            pk[c] = pack_bf16x2(pv.x, pv.y);
          }
          tmem_st_32x32b_x16(tS + 16 * gq, pk);
        }
        const float rsum = (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y) + (rs[2].x + rs[2].y) + (rs[3].x + rs[3].y);
        // O may be rescaled only once this item's previous P V into it has
        // completed (the first tile of an item starts a fresh O).  With one S
        // buffer per tile at most that P V is outstanding, and o_done's
        // parity names it.  With three buffers a single tile can have two
        // outstanding (its S was issued once the P V three back completed),
        // and a parity wait on o_done would then return on the older phase.
        // So there the wait is on pv_done of the previous P's buffer, which
        // has at most one use outstanding; P V products complete in issue
        // order, so that P V's completion implies every earlier one's.
        if (!corr_warps<D, WIN>() && it > w.lo[t] && __any_sync(0xffffffffu, alpha != 1.f)) {
          uint32_t pb = bar.o_done(t), pp = (n - 1) & 1;
          if constexpr (tri_s<D, WIN>()) {
            const int kp = k - (pair ? 2 : 1);
            pb = bar.pv_done(kp % 3);
            pp = (kp / 3) & 1;
          }
          if (!warp_wait(pb, pp)) {
            tmem_wait_st();
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t o[D];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_ld_32x32b_x32(tO + c * 32, &o[c * 32]);
          tmem_wait_ld();
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < D; e += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
            o[e] = __float_as_uint(v.x);
            o[e + 1] = __float_as_uint(v.y);
          }
#pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_st_32x32b_x32(tO + c * 32, &o[c * 32]);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(sb));
        l = l * alpha + rsum;
      }
      if (!ok) break;
      ks += pair ? 2 * w.ntiles : w.ntiles;
      // ------------------------------------------------------------ output
      // With a staging tile (D = 64), O goes out through shared memory: each
      // thread writes its normalised row (16-byte chunks XOR-swizzled by row),
      // then every warp copies whole rows with coalesced 16-byte stores, a
      // warp instruction covering 512 contiguous bytes.  The two query tiles
      // take the tile in turn, tile 0 then tile 1 of every item: use
      // u = 2 ni + t waits for the release of use u - 1.  (Measured at
      // 4x16x2048x64 and 2x16x8192x64: 5.5% faster than storing each row from
      // registers, where a warp instruction touches 32 rows.  At d = 96 and
      // 128 the SMEM left over would squeeze L1 and the gain vanished; with a
      // window it reversed.)
      if constexpr (kStagedOut) {
        const int u = 2 * ni + t;
        ++ni;
        if (u > 0 && !warp_wait(bar.o_free(), (u - 1) & 1)) {
          ok = false;
          break;
        }
      }
      // wait for this item's last P V (the next item's first P V into O needs
      // this warpgroup's first P of that item, so it cannot have started).
      // Three-buffer layout: up to three of this tile's P V products may still
      // be outstanding here (two for a tile of a pair), so, as for the
      // rescale, the wait is on pv_done of the tile's last P (ks already
      // counts this item's S products).
      if (w.lo[t] < w.hi[t]) {
        uint32_t eb = bar.o_done(t), ep = (n - 1) & 1;
        if constexpr (tri_s<D, WIN>()) {
          const int kl = ks - (pair ? 2 - t : 1);
          eb = bar.pv_done(kl % 3);
          ep = (kl / 3) & 1;
        }
        if (!warp_wait(eb, ep)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv_l = 1.f / (l + lc);
        if constexpr (kStagedOut) {
          const uint32_t srow = sOst + row * (2 * C::DP);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint32_t ch = c * 4 + q4;
              st_shared_v4(srow + ((ch ^ (row & 7)) << 4),
                           pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l),
                           pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l),
                           pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l),
                           pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l));
            }
          }
        } else {
          uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + (static_cast<size_t>(w.bh) * N + qi) * D * 2;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + c * 32, o);
            tmem_wait_ld();
            if (qi < N && !*abort_flag) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l);
                v.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l);
                v.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l);
                v.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l);
                st_global_v4(orow + (c * 4 + q4) * 16, v);
              }
            }
          }
        }
        if (p.lse != nullptr && qi < N) {
          const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;
          p.lse[static_cast<size_t>(w.bh) * N + qi] = (mref + __log2f(l)) * 0.69314718055994531f;
        }
        tc_fence_before();
        if constexpr (kStagedOut) {
          mbar_arrive(bar.o_staged(t));
          if (!warp_wait(bar.o_staged(t), no & 1)) {
            ok = false;
            break;
          }
          ++no;
          constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
          const int row0 = w.i0 + t * BR;
          const int nrows = min(BR, N - row0);
          uint8_t* obase = reinterpret_cast<uint8_t*>(p.o) + (static_cast<size_t>(w.bh) * N + row0) * D * 2;
          if (!*abort_flag) {
            for (int idx = row; idx < nrows * CHUNKS; idx += BR) {
              const int rr = idx / CHUNKS, ch = idx % CHUNKS;
              st_global_v4(obase + static_cast<size_t>(rr) * (D * 2) + ch * 16,
                           ld_shared_v4(sOst + rr * (2 * C::DP) + ((ch ^ (rr & 7)) << 4)));
            }
          }
        }
      }
      if constexpr (kStagedOut) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.o_free());
      }
    }
  };
  if constexpr (corr_warps<D, WIN>()) {
    if (warp >= 8) {
      regs_decrease<kRegsOther>();
      if (warp >= 12)
        role_correction();
      else if (warp == 9)
        role_tma();
      else if (warp == 8)
        role_mma();
    } else {
      regs_increase<kRegsSoftmax>();
      role_softmax();
    }
  } else {
    if (warp >= 10) {
      // warp 10 issues the P V products in the three-buffer layout; otherwise idle
      if (warp == 10) role_pv();
    } else if (warp == 9) {
      role_tma();
    } else if (warp == 8) {
      role_mma();
    } else {
      role_softmax();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

template <int D, bool WIN>
cudaError_t launch_d(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  using C = Cfg<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_bf16_sm103_kernel<D, WIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long pairs = static_cast<long long>((p.N + 2 * BR - 1) / (2 * BR)) * p.BH;
  if (2 * pairs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = static_cast<int>(pairs < sms ? pairs : sms);
  // Unmasked: a last round of pairs that fills at most half the CTAs runs as
  // single query tiles instead (twice the items, each half the work).
  long long n_pair = pairs, items = pairs;
  const long long rem = pairs % grid;
  if (!WIN && p.N > BR && rem > 0 && 2 * rem <= grid) {
    n_pair = pairs - rem;
    items = n_pair + 2 * rem;
  }
  fa_fwd_bf16_sm103_kernel<D, WIN><<<grid, threads_for<D, WIN>(), C::SMEM_BYTES, s>>>(
      m.q, m.k, m.v, p, static_cast<int>(items), static_cast<int>(n_pair));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16_tc(const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
  const bool win = p.window_r >= 0;
  // narrow bands (at most three key tiles per query tile): one query tile per
  // CTA, two CTAs per SM (fwd_bf16_win_sm103.cu)
  if (win && p.d != 256 && p.window_r <= 128) return launch_fwd_bf16_win(p, m, s);
  if (p.d == 128) return win ? launch_d<128, true>(p, m, s) : launch_d<128, false>(p, m, s);
  if (p.d == 64) return win ? launch_d<64, true>(p, m, s) : launch_d<64, false>(p, m, s);
  if (p.d == 96) return win ? launch_d<96, true>(p, m, s) : launch_d<96, false>(p, m, s);
  if (p.d == 256) return launch_fwd_bf16_d256(p, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
