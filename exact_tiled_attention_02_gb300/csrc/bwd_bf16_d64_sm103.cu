// bwd_bf16_d64_sm103.cu -- the attention backward's main kernel for head
// dimension 64 (bf16 in, fp32 accumulate, GB300 / sm_103a), with a schedule
// that overlaps the element-wise work of one query tile with the tensor work
// of the next.
//
// Same recomputation and the same five products per (key tile, query tile)
// step as the general kernel in bwd_bf16_sm103.cu ("Flash attention and
// efficient attention -- Hinglish notes", "Backward Pass: Recomputation": P
// is rebuilt from Q, K and the forward's logsumexp, never read; the gradient
// formulas are the derivative of the forward definition):
//   S'^T  = K Q_i^T - lse_i / scale,  P^T = exp2(S'^T scale log2e)
//   dP'^T = V dO_i^T - D_i,           dS^T = P^T o dP'^T
//   dV += P^T dO_i,  dK += dS^T Q_i,  dQ_i = dS K   (dQ added into an fp32
//   accumulator by TMA reductions; dK scaled and both cast at the end)
//
// Two things differ from the general kernel.
//
// (1) The per-query terms -lse_i / scale and -D_i are added by the tensor
// core, as one more K = 16 step of S^T and of dP^T (a (1, 1, 1, 0...) row per
// key times three bf16 terms per query that sum to the fp32 value; the prep
// kernel writes the terms).  The element-wise passes then read nothing but
// TMEM.  Loading a 64-value vector per thread from shared memory instead (a
// broadcast, 512 bytes of register write-back per warp instruction) held
// each of those passes to the shared-memory return bandwidth: measured
// ~520 cycles per pass for the vector alone, with ~1660 cycles of tensor work
// per step.
//
// (2) The schedule, which d = 64 makes possible.  At d = 128 the four
// accumulators S^T, dP^T, dV, dK fill the 512 TMEM columns, so dQ has to
// borrow the S^T columns and the next S^T waits for dQ to be read out: every
// step runs S^T -> P -> dS -> dQ -> read-out back to back.  At d = 64, dV and
// dK take 64 columns each and dQ gets 64 columns of its own:
//   [0,128) S^T / P^T   [128,256) dP^T / dS^T   [256,320) dV   [320,384) dK
//   [384,448) dQ
// so, per step i, the MMA threads issue
//   dV_i (once P_i is in TMEM) and S^T_{i+1}; on a second thread dK_i (once
//   dS_i is in TMEM) and dP^T_{i+1}; on a third dQ_i (once dS_i is in shared
//   memory)
// and the compute warpgroups run dS_i, then P_{i+1} (its S^T_{i+1} already
// computed), then the read-out of dQ_i: the exponentials of the next tile
// overlap this tile's dQ and dK products.  dQ_i and dK_i go out from two
// threads once dS_i is in place, so dQ_i need not queue behind dK_i before
// the warpgroups come to read it.  Shared memory also has
// room at d = 64 for a dedicated dQ staging tile and a three-stage Q/dO
// ring, so the ring is refilled as soon as dK_i has read Q_i, independently
// of the dQ reductions.
//
// Warp roles (384 threads): warps 0-3 and 4-7 are the two compute
// warpgroups (query columns 0-63 / 64-127 of every tile; thread t owns key
// row t == TMEM lane t, and for the dQ read-out query row t, warpgroup g
// taking d columns [32g, 32g + 32)); warp 8 owns TMEM and issues dV and S^T;
// warp 10 issues dK and dP^T, warp 11 dQ (measured at 2x16x8192x64: a
// second issuing thread, for dQ, dK and dP^T, 2.6% faster than one; dQ on a
// third, 1.355 -> 1.324 ms); warp 9 is the TMA producer (loads, dQ
// reductions).
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int BM = 128;  // query rows per step
constexpr int BN = 128;  // keys per CTA
constexpr int D = 64;
constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 320, TM_DQ = 384;
constexpr int STAGES = 3;
constexpr int TILE_BYTES = 128 * D * 2;          // bf16 [128][64]: one 128-byte-swizzled box
constexpr int STAGE_BYTES = 2 * TILE_BYTES;      // Q_i then dO_i
constexpr int DST_BYTES = BN * BM * 2;           // bf16 dS^T [128 keys][128 queries], two boxes
constexpr int DST_BOX = 128 * 128;               // one [128][64] bf16 box
constexpr int OST_BOX = BM * 32 * 4;             // fp32 dQ staging box [128 queries][32 d], 128-byte swizzled
// The row terms -lse_q / scale and -D_q enter S^T and dP^T as one extra K = 16
// step each: A = a [128 keys][16] tile whose rows are (1, 1, 1, 0...), B = the
// query tile's rows (t1, t2, t3, 0...), three bf16 terms summing to the fp32
// value.  Both operands are K-major without swizzle: 16-byte rows (the first
// core matrix of each 8-row group, groups 128 bytes apart) and a second core
// matrix (elements 8-15) that is a shared 2 KB block of zeros.
constexpr int AUG_BYTES = BM * 16;
// The small operands come first, each below the shared zero block (a
// descriptor's byte offsets are unsigned); the 1024-aligned tiles follow.
constexpr int OFF_AUG = 0;                                  // per stage: Q's terms, then dO's
constexpr int OFF_ONES = OFF_AUG + STAGES * 2 * AUG_BYTES;  // the (1, 1, 1, 0...) rows
constexpr int OFF_ZERO = OFF_ONES + AUG_BYTES;              // elements 8-15 of every such operand
constexpr int OFF_K = OFF_ZERO + AUG_BYTES;
constexpr int OFF_V = OFF_K + TILE_BYTES;
constexpr int OFF_STAGE = OFF_V + TILE_BYTES;
constexpr int OFF_DST = OFF_STAGE + STAGES * STAGE_BYTES;
constexpr int OFF_OST = OFF_DST + DST_BYTES;
constexpr int OFF_BAR = OFF_OST + 2 * OST_BOX;
// kv_full, st_full[3], stage_free[3], s_full, dp_full, p_full, ds_full, dq_full, staged, ost_free, fin, drain,
// drain2, drain3
constexpr int NBAR = 1 + 2 * STAGES + 11;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
// the whole 227 KB: every address an MMA operand descriptor can form (16
// groups of either offset) stays inside the allocation
constexpr int SMEM_BYTES = 227 * 1024;
static_assert(SMEM_USED + 1024 <= SMEM_BYTES, "shared memory budget");
static_assert(OFF_AUG + 15 * (OFF_ZERO - OFF_AUG) + 256 + 1024 <= SMEM_BYTES, "operand offsets in bounds");
static_assert(OFF_K % 1024 == 0 && OFF_STAGE % 1024 == 0 && OFF_DST % 1024 == 0 && OFF_OST % 1024 == 0,
              "swizzled tiles 1024-aligned");

struct Bars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t st_full(int s) const { return base + 8 * (1 + s); }  // Q_i, dO_i and their terms
  __device__ uint32_t stage_free(int s) const { return base + 8 * (1 + STAGES + s); }
  __device__ uint32_t at(int k) const { return base + 8 * (1 + 2 * STAGES + k); }
  __device__ uint32_t s_full() const { return at(0); }
  __device__ uint32_t dp_full() const { return at(1); }
  __device__ uint32_t p_full() const { return at(2); }
  __device__ uint32_t ds_full() const { return at(3); }
  __device__ uint32_t dq_full() const { return at(4); }
  __device__ uint32_t staged() const { return at(5); }
  __device__ uint32_t ost_free() const { return at(6); }
  __device__ uint32_t fin() const { return at(7); }
  __device__ uint32_t drain() const { return at(8); }
  __device__ uint32_t drain2() const { return at(9); }
  __device__ uint32_t drain3() const { return at(10); }
};

__host__ __device__ __forceinline__ int npad128(int n) { return (n + 127) & ~127; }


// Shared-memory descriptor of a K-major operand without swizzle: 8-row groups
// of 16-byte rows `sbo` bytes apart, the core matrix of the next 8 K-elements
// `lbo` bytes after the first.
__device__ __forceinline__ uint64_t sdesc_noswz(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version (tcgen05); swizzle mode 0: none
  return d;
}

__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_bf16_d64_sm103_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                                 const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                                 const __grid_constant__ CUtensorMap tmdq, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + SMEM_USED > static_cast<uint32_t>(SMEM_BYTES)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sK = sb + OFF_K, sV = sb + OFF_V, sStage = sb + OFF_STAGE, sDS = sb + OFF_DST, sOst = sb + OFF_OST,
                 sAug = sb + OFF_AUG, sOnes = sb + OFF_ONES, sZero = sb + OFF_ZERO;
  const Bars bar{sb + OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, r = p.window_r;
  const int nkt = (N + BN - 1) / BN;
  // CTAs past n_full take one half of a split key tile's query tiles each
  int tile = static_cast<int>(blockIdx.x), half = -1;
  if (tile >= p.n_full) {
    half = (tile - p.n_full) & 1;
    tile = p.n_full + ((tile - p.n_full) >> 1);
  }
  const int bh = tile / nkt;
  const int k0 = (tile % nkt) * BN;
  const int np = npad128(N);
  int t_lo = 0, t_hi = (N + BM - 1) / BM;  // query tiles that can see this key tile
  if (r >= 0) {
    t_lo = max(0, k0 - r) / BM;
    t_hi = (min(N, k0 + BN + r) + BM - 1) / BM;
  }
  if (half >= 0) {
    const int mid = t_lo + (t_hi - t_lo) / 2;
    if (half == 0)
      t_hi = mid;
    else
      t_lo = mid;
  }
  const int nsteps = t_hi - t_lo;

  if (threadIdx.x == 0) {
    mbar_init(bar.kv_full(), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar.st_full(s), 1);
      mbar_init(bar.stage_free(s), 2);  // commits after dV_i and after dK_i, the stage's last readers
    }
    mbar_init(bar.s_full(), 1);
    mbar_init(bar.dp_full(), 1);
    mbar_init(bar.p_full(), 8);  // one arrive per compute warp
    mbar_init(bar.ds_full(), 8);
    mbar_init(bar.dq_full(), 1);
    mbar_init(bar.staged(), 8);
    mbar_init(bar.ost_free(), 1);  // the producer, once a reduction has read the staging tile
    mbar_init(bar.fin(), 3);  // one commit per MMA-issuing thread
    mbar_init(bar.drain(), 1);
    mbar_init(bar.drain2(), 1);
    mbar_init(bar.drain3(), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  for (int idx = threadIdx.x; idx < BM; idx += kThreads) {
    // bf16 1.0 = 0x3f80
    st_shared_v4(sOnes + idx * 16, 0x3f803f80u, 0x3f80u, 0u, 0u);
    st_shared_v4(sZero + idx * 16, 0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();  // read by tcgen05.mma (async proxy)
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
  };

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmq);
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      prefetch_tensormap(&tmdo);
      prefetch_tensormap(&tmdq);
      mbar_arrive_expect_tx(bar.kv_full(), 2 * TILE_BYTES);
      tma_load_3d(sK, &tmk, bar.kv_full(), 0, k0, bh);
      tma_load_3d(sV, &tmv, bar.kv_full(), 0, k0, bh);
      // tile `it` into stage it % STAGES: Q_it with its -lse / scale terms, and dO_it with its -D terms
      auto load = [&](int it) {
        const int st = it % STAGES;
        const int q0 = (t_lo + it) * BM;
        const uint32_t base = sStage + st * STAGE_BYTES;
        const uint32_t aug = sAug + st * 2 * AUG_BYTES;
        mbar_arrive_expect_tx(bar.st_full(st), 2 * TILE_BYTES + 2 * AUG_BYTES);
        tma_load_3d(base, &tmq, bar.st_full(st), 0, q0, bh);
        const size_t vrow = static_cast<size_t>(bh) * np + q0;
        bulk_load(aug, reinterpret_cast<const uint8_t*>(p.lse2) + vrow * 16, AUG_BYTES, bar.st_full(st));
        bulk_load(aug + AUG_BYTES, reinterpret_cast<const uint8_t*>(p.dsum) + vrow * 16, AUG_BYTES, bar.st_full(st));
        tma_load_3d(base + TILE_BYTES, &tmdo, bar.st_full(st), 0, q0, bh);
      };
      int loaded = 0;
      for (; loaded < STAGES && loaded < nsteps; ++loaded) load(loaded);
      for (int it = 0; it < nsteps; ++it) {
        // the stage of tile it takes tile it + STAGES once dK_it has read Q_it
        if (loaded < nsteps) {
          if (!mbar_wait_backoff(bar.stage_free(it % STAGES), (it / STAGES) & 1, wc)) break;
          load(loaded);
          ++loaded;
        }
        // dQ_it, staged by the compute warpgroups as two fp32 [128][32] boxes
        if (!mbar_wait_backoff(bar.staged(), it & 1, wc)) break;
        const int q0 = (t_lo + it) * BM;
        tma_reduce_add_3d(&tmdq, sOst, 0, q0, bh);
        tma_reduce_add_3d(&tmdq, sOst + OST_BOX, 32, q0, bh);
        bulk_commit_group();
        bulk_wait_read_all();
        mbar_arrive(bar.ost_free());
      }
      bulk_wait_all();  // reductions complete before the CTA exits
      if (*abort_flag) {
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.kv_full(), 0, drain);
        for (int it = max(0, loaded - STAGES); it < loaded; ++it) {
          mbar_wait(bar.st_full(it % STAGES), (it / STAGES) & 1, drain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 8 || warp == 10 || warp == 11) {
    // ----------------------------------------------------------------- MMA
    // Three issuing threads on three SM sub-partitions (each shares its
    // sub-partition with two compute warps, whose instructions delay the
    // issue; and issuing a tcgen05.mma takes about as long as executing one
    // of N = 64): warp 8 issues dV_i and S^T_{i+1}, warp 10 dK_i and
    // dP^T_{i+1}, warp 11 dQ_i.  None writes what another's products read,
    // and each thread's products run in its issue order; the stage is free
    // once warps 8 and 10 have committed (stage_free counts two: dQ does not
    // read the stage), and the epilogue once all three have (fin).
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);  // both operands K-major
      constexpr uint32_t id_kb = idesc_bf16_f32(128, D, 0, 1);    // A from TMEM, B MN-major, N = 64
      constexpr uint32_t id_mm = idesc_bf16_f32(128, D, 1, 1);    // both MN-major (dS, K), N = 64
      // P^T / dS^T of query columns 16kk.. sit at TMEM column 8kk, or 64 + 8(kk - 4)
      auto pcol = [](int kk) { return static_cast<uint32_t>(kk < 4 ? 8 * kk : 64 + 8 * (kk - 4)); };
      bool ok = mbar_wait2(bar.kv_full(), 0, bar.st_full(0), 0, wc);
      if (ok) tc_fence_after();
      if (warp == 11) {
        // dQ_i = dS K into its own columns, once dS_i is in shared memory (the
        // warpgroups read dQ_{i-1} out before computing dS_i: ds_full also
        // frees the columns)
        for (int i = 0; ok && i < nsteps; ++i) {
          if (!mbar_wait(bar.ds_full(), i & 1, wc)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_bf16_ss(tmem + TM_DQ, sdesc_sw128(sDS + kk * 2048, DST_BOX, 1024),
                        sdesc_sw128(sK + kk * 2048, TILE_BYTES, 1024), id_mm, kk > 0);
          mma_commit(bar.dq_full());
        }
        mma_commit(bar.fin());
        mma_commit(bar.drain3());
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.drain3(), 0, drain);
      } else if (warp == 8) {
        // S^T_i = K Q_i^T (stage i % STAGES resident)
        auto issue_s = [&](int i) {
          const int st = i % STAGES;
          const uint32_t qb = sStage + st * STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss(tmem + TM_S, sdesc_sw128(sK + kk * 32, 16, 1024), sdesc_sw128(qb + kk * 32, 16, 1024), id_kk,
                        kk > 0);
          const uint32_t qa = sAug + st * 2 * AUG_BYTES;  // + (1, 1, 1) . (-lse_q / scale terms)
          mma_bf16_ss(tmem + TM_S, sdesc_noswz(sOnes, sZero - sOnes, 128), sdesc_noswz(qa, sZero - qa, 128), id_kk,
                      1);
          mma_commit(bar.s_full());
        };
        if (ok) issue_s(0);
        for (int i = 0; ok && i < nsteps; ++i) {
          const int st = i % STAGES;
          const uint32_t ph = i & 1;
          const uint32_t qb = sStage + st * STAGE_BYTES;
          const bool more = i + 1 < nsteps;
          // dV += P^T dO_i, then the next S^T into the columns P^T_i leaves (P_i
          // in TMEM and, with it, stage i + 1 resident)
          if (more ? !mbar_wait2(bar.p_full(), ph, bar.st_full((i + 1) % STAGES), ((i + 1) / STAGES) & 1, wc)
                   : !mbar_wait(bar.p_full(), ph, wc))
            break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_bf16_ts(tmem + TM_DV, tmem + TM_S + pcol(kk),
                        sdesc_sw128(qb + TILE_BYTES + kk * 2048, TILE_BYTES, 1024), id_kb, (i > 0 || kk > 0));
          mma_commit(bar.stage_free(st));  // dO_i's last reader
          if (more) issue_s(i + 1);
        }
        mma_commit(bar.fin());
        mma_commit(bar.drain());
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.drain(), 0, drain);
      } else {
        // dP^T_i = V dO_i^T (stage i % STAGES resident)
        auto issue_dp = [&](int i) {
          const int st = i % STAGES;
          const uint32_t ob = sStage + st * STAGE_BYTES + TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss(tmem + TM_DP, sdesc_sw128(sV + kk * 32, 16, 1024), sdesc_sw128(ob + kk * 32, 16, 1024), id_kk,
                        kk > 0);
          const uint32_t oa = sAug + st * 2 * AUG_BYTES + AUG_BYTES;  // + (1, 1, 1) . (-D_q terms)
          mma_bf16_ss(tmem + TM_DP, sdesc_noswz(sOnes, sZero - sOnes, 128), sdesc_noswz(oa, sZero - oa, 128), id_kk,
                      1);
          mma_commit(bar.dp_full());
        };
        if (ok) issue_dp(0);
        for (int i = 0; ok && i < nsteps; ++i) {
          const int st = i % STAGES;
          const uint32_t ph = i & 1;
          const uint32_t qb = sStage + st * STAGE_BYTES;
          const bool more = i + 1 < nsteps;
          // (dQ_i is warp 11's.)  dK += dS^T Q_i (Q_i's last reader), then the
          // next dP^T into the columns dS^T_i leaves
          if (more ? !mbar_wait2(bar.ds_full(), ph, bar.st_full((i + 1) % STAGES), ((i + 1) / STAGES) & 1, wc)
                   : !mbar_wait(bar.ds_full(), ph, wc))
            break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_bf16_ts(tmem + TM_DK, tmem + TM_DP + pcol(kk), sdesc_sw128(qb + kk * 2048, TILE_BYTES, 1024), id_kb,
                        (i > 0 || kk > 0));
          mma_commit(bar.stage_free(st));
          if (more) issue_dp(i + 1);
        }
        mma_commit(bar.fin());
        mma_commit(bar.drain2());
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.drain2(), 0, drain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- compute warpgroups
    const int g = warp >> 2;            // query columns [64g, 64g + 64) of every tile
    const int row = threadIdx.x & 127;  // key row == TMEM lane (query row for the dQ read-out)
    const int kj = k0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tS = tl + TM_S + 64 * g, tDP = tl + TM_DP + 64 * g;
    // this thread's row of its dS^T box and of its dQ staging box (both 128-byte
    // swizzled and 1024-aligned: 16-byte chunk c of the row sits at row ^ (c << 4))
    const uint32_t dsrow = sDS + g * DST_BOX + row * 128 + ((row & 7) << 4);
    const uint32_t strow = sOst + g * OST_BOX + row * 128 + ((row & 7) << 4);
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    float pr[64];  // P of the current step, kept for dS
    // ---- P^T_i = exp2((S^T_i - lse / scale) * scale * log2e), to TMEM for dV
    //      (S^T_i already holds the -lse / scale term: no per-column vector)
    auto p_phase = [&](int i) -> bool {
      if (!warp_wait(bar.s_full(), i & 1)) return false;
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_32x32b_x32(tS, &sv[0]);
      tmem_ld_32x32b_x32(tS + 32, &sv[32]);
      tmem_wait_ld();
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float2 x0 = __fmul2_rn(make_float2(__uint_as_float(sv[4 * c4]), __uint_as_float(sv[4 * c4 + 1])), sl2);
        const float2 x1 = __fmul2_rn(make_float2(__uint_as_float(sv[4 * c4 + 2]), __uint_as_float(sv[4 * c4 + 3])), sl2);
        pr[4 * c4] = ex2_approx(x0.x);
        pr[4 * c4 + 1] = ex2_approx(x0.y);
        pr[4 * c4 + 2] = ex2_approx(x1.x);
        pr[4 * c4 + 3] = ex2_approx(x1.y);
      }
      const int q0 = (t_lo + i) * BM + 64 * g;  // first query column of this warpgroup
      if (r >= 0 && !(q0 >= kj - r && q0 + 63 <= kj + r)) {
        // window: the queries that see key kj form one contiguous column range [lo, hi)
        const int lo = max(0, kj - r - q0), hi = min(64, kj + r + 1 - q0);
        const unsigned span = hi > lo ? static_cast<unsigned>(hi - lo) : 0u;
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = (static_cast<unsigned>(c - lo) < span) ? pr[c] : 0.f;
      }
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(pr[2 * c], pr[2 * c + 1]);
      tmem_st_32x32b_x32(tS, pk);  // P^T over this warpgroup's first 32 S^T columns
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full());
      return true;
    };
    // Key rows past N hold zeros (TMA zero fill): their P and dS are finite and
    // meet K = 0 in dQ; their dK / dV rows are never stored.  No mask needed.
    // pass j: dS of tile j - 1, P of tile j, the dQ read-out of tile j - 1.
    // (Only the last pass skips P and it leaves the loop, so P is dead after
    // each dS on every path: it need not share the registers with dP.)
    bool ok = true;
    for (int j = 0;; ++j) {
      const bool last = j == nsteps;
      const int i = j - 1;
      const uint32_t ph = i & 1;
      // ---- dS^T_i = P^T o (dP^T - D), to TMEM (for dK) and shared memory (for
      //      dQ; the previous dQ has completed, its read-out waited for it).
      //      dP^T_i already holds the -D term.
      if (j > 0) {
      if (!warp_wait(bar.dp_full(), ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t dpv[64];
        tmem_ld_32x32b_x32(tDP, &dpv[0]);
        tmem_ld_32x32b_x32(tDP + 32, &dpv[32]);
        tmem_wait_ld();
        uint32_t dk[32];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float2 t0 = make_float2(__uint_as_float(dpv[4 * c4]), __uint_as_float(dpv[4 * c4 + 1]));
          const float2 t1 = make_float2(__uint_as_float(dpv[4 * c4 + 2]), __uint_as_float(dpv[4 * c4 + 3]));
          const float2 d0 = __fmul2_rn(make_float2(pr[4 * c4], pr[4 * c4 + 1]), t0);
          const float2 d1 = __fmul2_rn(make_float2(pr[4 * c4 + 2], pr[4 * c4 + 3]), t1);
          dk[2 * c4] = pack_bf16x2(d0.x, d0.y);
          dk[2 * c4 + 1] = pack_bf16x2(d1.x, d1.y);
        }
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          st_shared_v4(dsrow ^ (c8 << 4), dk[4 * c8], dk[4 * c8 + 1], dk[4 * c8 + 2], dk[4 * c8 + 3]);
        tmem_st_32x32b_x32(tDP, dk);  // dS^T over this warpgroup's first 32 dP^T columns
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.ds_full());
      }

      // ---- the next tile's P while dK_i and dQ_i run
      if (!last && !p_phase(j)) {
        ok = false;
        break;
      }
      if (j == 0) {
        if (last) break;
        continue;
      }

      // ---- dQ_i read-out (thread = query row, warpgroup g takes d columns
      //      [32g, 32g + 32)), staged as fp32 box g of the staging tile
      if (!warp_wait(bar.dq_full(), ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t qv[32];
      tmem_ld_32x32b_x32(tl + TM_DQ + 32 * g, qv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (i > 0 && !warp_wait(bar.ost_free(), (i - 1) & 1)) {  // the previous reduction has read the tile
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) st_shared_v4(strow ^ (c << 4), qv[4 * c], qv[4 * c + 1], qv[4 * c + 2], qv[4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.staged());
      if (last) break;
    }

    // ------------------------------------------------------------ epilogue
    // warpgroup 0 writes dV, warpgroup 1 writes scale * dK, each staged as a
    // bf16 [128 keys][64] tile over K (dV) or V (dK), which nothing reads once
    // every product has completed
    const bool have = ok && warp_wait(bar.fin(), 0);
    const uint32_t stage_out = g == 0 ? sK : sV;
    if (have && half >= 0) {
      // one half of a split key tile: add this row's fp32 values into the
      // partial rows (two addends into zeroed memory: order-independent)
      tc_fence_after();
      const uint32_t tcol = g == 0 ? TM_DV : TM_DK;
      const float mul = g == 0 ? 1.f : p.scale;
      float* dst = p.kv_part + ((static_cast<size_t>(tile - p.n_full) * 2 + g) * BN + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tl + tcol + c * 32, v);
        tmem_wait_ld();
        if (k0 + row < N) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            red_add_v4_f32(dst + c * 32 + 4 * e, __uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                           __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
        }
      }
    } else if (have) {
      tc_fence_after();
      const uint32_t tcol = g == 0 ? TM_DV : TM_DK;
      const float mul = g == 0 ? 1.f : p.scale;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tl + tcol + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c16 = c * 4 + q4;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * e]) * mul, __uint_as_float(v[q4 * 8 + 2 * e + 1]) * mul);
          st_shared_v4(stage_out + row * (2 * D) + ((c16 ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
      }
    }
    tc_fence_before();
    named_bar_sync(1 + g, 128);
    if (have && half < 0 && !*abort_flag) {
      uint8_t* gout = reinterpret_cast<uint8_t*>(g == 0 ? p.dv : p.dk) + (static_cast<size_t>(bh) * N + k0) * D * 2;
      constexpr int CHUNKS = D / 8;
      for (int idx = row; idx < BN * CHUNKS; idx += 128) {
        const int rr = idx / CHUNKS, c16 = idx % CHUNKS;
        if (k0 + rr < N)
          st_global_v4(gout + static_cast<size_t>(rr) * (2 * D) + c16 * 16,
                       ld_shared_v4(stage_out + rr * (2 * D) + ((c16 ^ (rr & 7)) << 4)));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_bwd_main_d64(const BwdParams& p, const BwdMaps& m, unsigned grid, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(fa_bwd_bf16_d64_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  fa_bwd_bf16_d64_sm103_kernel<<<grid, kThreads, SMEM_BYTES, s>>>(m.q, m.k, m.v, m.dO, m.dq_acc, p);
  return cudaGetLastError();
}

}  // namespace fa
