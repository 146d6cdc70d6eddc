// fwd.cu -- fused attention forward for sm_103a.
//
// fwd_kernel: a persistent CTA per SM walks work items, each one 128-row
// query tile of one (batch, q head) and, for head_dim 512, one half of the
// value columns (the "D-split": both halves recompute S = Q K^T over the full
// head dim, each accumulates half of O, so O never needs more than 256 TMEM
// columns). The same kernel serves head_dim 256, 512 and the asymmetric pair
// Q/K 192, V/O 128.
//
// Roles (256 threads):
//   warp 0      TMA producer: Q once, then K/V tiles through a ring of 32 KB
//               stages, in exactly the order the MMA warp consumes them. A
//               K tile takes DQK/128 stages of 128 keys x 128 columns, and a
//               final half-filled one (64 columns) when DQK is an odd
//               multiple of 64.
//   warp 1      TMEM allocator and MMA issuer (one elected thread):
//                 S_j = Q K_j^T  (SS MMA, fp32 in TMEM, double-buffered)
//                 O  += P_j V_j  (TS MMA, P read from TMEM)
//               issued as S_0, S_1, PV_0, S_2, PV_1, ... so that S_{j+1} runs
//               on the tensor pipe while the softmax warps work on S_j.
//   warps 4-7   softmax: one thread per query row. Loads S_j from TMEM,
//               masks edge tiles, keeps a running row max m and sum l,
//               writes P_j = exp2((S_j - m) * scale * log2 e) as 16-bit values
//               back into the S_j columns, and rescales O in TMEM only when
//               the max grew by more than 2^8 (otherwise P stays <= 256).
//               Epilogue: O / l to global memory, LSE = m*scale + ln l.
// The TMEM plan: O at columns [0, DV), S/P buffers at DV and DV+128; with
// DV <= 256 this fits the 512 columns of one SM.
#include <algorithm>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"
#include "kernels.h"

namespace sdpa {

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int STAGE_BYTES = 32768;
  static constexpr int Q_BYTES = DQK * 256;  // 128 rows x DQK x 2 bytes
  static_assert(DQK % 64 == 0 && DV % 64 == 0, "head dims are whole 64-column swizzle atoms");
  static constexpr int NSTAGES = DQK <= 192 ? 5 : (DQK == 256 ? 5 : 3);
  static constexpr int KST = (DQK + 127) / 128;            // K stages per tile (128 keys x up to 128 d each)
  // 64-column atoms of K stage kb (two, or one for the last stage of DQK = 192)
  static __device__ __forceinline__ constexpr int k_atoms(int kb) { return DQK / 64 - 2 * kb >= 2 ? 2 : 1; }
  static constexpr int VROWS = STAGE_BYTES / (DV * 2);     // keys per V stage
  static constexpr int VST = BN / VROWS;                   // V stages per tile
  static constexpr int V_ATOM_BYTES = VROWS * 128;         // one 64-column swizzle atom of a V stage
  static constexpr int TMEM_O = 0, TMEM_S = DV;
  static constexpr int NBARS = 2 * NSTAGES + 9;
  static constexpr int SMEM_BYTES = 1024 + Q_BYTES + NSTAGES * STAGE_BYTES + NBARS * 8 + 16;
};

// A work item of the order: a query tile (heaviest, i.e. last, first; GQA
// heads adjacent) and the value-column split this CTA accumulates.
struct FwdItem {
  int split, q0, q_last, t_lo, n, qhead, khead;
  SeqInfo si;
  KeyRange kr;
};

template <int DQK, int DV>
__device__ __forceinline__ bool fwd_item(const FwdParams& p, int idx, FwdItem& t) {
  using C = FwdCfg<DQK, DV>;
  const Geom& g = p.g;
  t.split = idx % p.dv_splits;
  idx /= p.dv_splits;
  const int h = idx % g.hq;
  idx /= g.hq;
  const int b = idx % g.batch;
  idx /= g.batch;
  t.q0 = (p.n_q_tiles - 1 - idx) * C::BM;
  t.si = seq_info(g, b);
  if (t.q0 >= t.si.lq) return false;
  t.kr = key_range(g, t.si.lq, t.si.lk);
  t.q_last = min(t.q0 + C::BM - 1, t.si.lq - 1);
  const int kv_lo = t.kr.lo(t.q0), kv_hi = t.kr.hi(t.q_last);
  t.t_lo = kv_lo / C::BN;
  t.n = (kv_hi > kv_lo) ? (kv_hi + C::BN - 1) / C::BN - t.t_lo : 0;
  t.qhead = t.si.qhead0 + h;
  t.khead = t.si.khead0 + h / (g.hq / g.hkv);
  return true;
}

// Persistent: CTA c takes the items c, c + gridDim.x, ... of the order and
// every role walks that same sequence. Barrier phases run on across items
// (S/P by step, O by P V, Q and the item's end by item). The next item's Q
// is loaded as soon as this item's last S is done (q_free); its first P V,
// which overwrites O, waits for the epilogue to have read O (o_free), so the
// next item's first S MMAs run during this item's epilogue.
template <int DQK, int DV, bool BF16>
__global__ void __launch_bounds__(256, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using C = FwdCfg<DQK, DV>;
  using E = Elem<BF16>;
  const Geom& g = p.g;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;
  const int total = p.total_tiles;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
  uint8_t* sQ = smem;
  uint8_t* sStage = smem + C::Q_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + C::NSTAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::NSTAGES;
  uint64_t* bar_q = empty + C::NSTAGES;
  uint64_t* bar_s = bar_q + 1;  // [2]
  uint64_t* bar_p = bar_s + 2;  // [2]
  uint64_t* bar_o = bar_p + 2;
  uint64_t* bar_drain = bar_o + 1;
  uint64_t* q_free = bar_drain + 1;  // an item's last S MMA is done: Q may be replaced
  uint64_t* o_free = q_free + 1;     // the epilogue has read O out of TMEM
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(o_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSTAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(bar_q, 1);
    mbar_init(&bar_s[0], 1);
    mbar_init(&bar_s[1], 1);
    mbar_init(&bar_p[0], 128);
    mbar_init(&bar_p[1], 128);
    mbar_init(bar_o, 1);
    mbar_init(bar_drain, 1);
    mbar_init(q_free, 1);
    mbar_init(o_free, 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int c = 0, nq = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < total && ok; idx += gridDim.x) {
        FwdItem t;
        if (!fwd_item<DQK, DV>(p, idx, t) || t.n == 0) continue;
        if (nq > 0 && !mbar_wait(q_free, (nq - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar_q, C::Q_BYTES);
        for (int a = 0; a < DQK / 64; ++a)
          tma_load_3d(&tmQ, bar_q, sQ + a * 16384, a * 64, t.qhead, t.si.qrow0 + t.q0);
        ++nq;
        auto next_slot = [&](int& slot, uint32_t bytes) -> bool {
          slot = c % C::NSTAGES;
          const uint32_t ph = (c / C::NSTAGES) & 1;
          if (!mbar_wait(&empty[slot], ph ^ 1, abort_flag)) return false;
          mbar_arrive_expect_tx(&full[slot], bytes);
          return true;
        };
        auto load_k = [&](int j) -> bool {
          const int key0 = t.si.krow0 + (t.t_lo + j) * C::BN;
          for (int kb = 0; kb < C::KST; ++kb, ++c) {
            int slot;
            const int atoms = C::k_atoms(kb);
            if (!next_slot(slot, atoms * 16384)) return false;
            uint8_t* dst = sStage + slot * C::STAGE_BYTES;
            tma_load_3d(&tmK, &full[slot], dst, kb * 128, t.khead, key0);
            if (atoms == 2) tma_load_3d(&tmK, &full[slot], dst + 16384, kb * 128 + 64, t.khead, key0);
          }
          return true;
        };
        auto load_v = [&](int j) -> bool {
          for (int vs = 0; vs < C::VST; ++vs, ++c) {
            int slot;
            if (!next_slot(slot, C::STAGE_BYTES)) return false;
            uint8_t* dst = sStage + slot * C::STAGE_BYTES;
            const int key0 = t.si.krow0 + (t.t_lo + j) * C::BN + vs * C::VROWS;
            for (int a = 0; a < DV / 64; ++a)
              tma_load_3d(&tmV, &full[slot], dst + a * C::V_ATOM_BYTES, t.split * DV + a * 64, t.khead, key0);
          }
          return true;
        };
        for (int j = 0; j < t.n && ok; ++j) {
          ok = load_k(j);
          if (ok && j >= 1) ok = load_v(j - 1);
        }
        if (ok) ok = load_v(t.n - 1);
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
      // Every issued copy must land before the CTA exits: the last NSTAGES
      // stages (or fewer) are the only ones that can still be in flight.
      const int first = c > C::NSTAGES ? c - C::NSTAGES : 0;
      for (int k = first; k < c; ++k) mbar_wait_drain(&full[k % C::NSTAGES], (k / C::NSTAGES) & 1);
      if (nq > 0) mbar_wait_drain(bar_q, (nq - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t IDESC_S = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t IDESC_O = idesc_f16(128, DV, BF16, false, true);
      int c = 0, nq = 0, gs = 0;  // ring stages, items with keys, steps of earlier items
      bool ok = true;
      const uint32_t q_base = smem_u32(sQ);
      for (int idx = blockIdx.x; idx < total && ok; idx += gridDim.x) {
        FwdItem t;
        if (!fwd_item<DQK, DV>(p, idx, t) || t.n == 0) continue;
        const int n = t.n;
        if (!mbar_wait(bar_q, nq & 1, abort_flag)) {
          ok = false;
          break;
        }
        ++nq;
        tc_fence_after();
        auto mma_s = [&](int j) -> bool {
          const int sj = gs + j;
          const uint32_t d = tmem + C::TMEM_S + (sj & 1) * 128;
          for (int kb = 0; kb < C::KST; ++kb, ++c) {
            const int slot = c % C::NSTAGES;
            if (!mbar_wait(&full[slot], (c / C::NSTAGES) & 1, abort_flag)) return false;
            tc_fence_after();
            const uint32_t k_base = smem_u32(sStage + slot * C::STAGE_BYTES);
            const uint32_t qa = q_base + kb * 2 * 16384;
            const int n_ks = 4 * C::k_atoms(kb);  // 16-column K steps held by this stage
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              if (ks >= n_ks) break;
              const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
              mma_ss(d, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(k_base + off, 16, 1024), IDESC_S,
                     (kb | ks) != 0);
            }
            mma_commit(&empty[slot]);
          }
          mma_commit(&bar_s[sj & 1]);
          if (j == n - 1) mma_commit(q_free);  // the item's last read of Q
          return true;
        };
        auto mma_o = [&](int j) -> bool {
          const int sj = gs + j;
          if (j == 0 && nq > 1) {  // O still holds the previous item until its epilogue read it
            if (!mbar_wait(o_free, (nq - 2) & 1, abort_flag)) return false;
          }
          if (!mbar_wait(&bar_p[sj & 1], (sj >> 1) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t pcol = tmem + C::TMEM_S + (sj & 1) * 128;
          for (int vs = 0; vs < C::VST; ++vs, ++c) {
            const int slot = c % C::NSTAGES;
            if (!mbar_wait(&full[slot], (c / C::NSTAGES) & 1, abort_flag)) return false;
            tc_fence_after();
            const uint32_t v_base = smem_u32(sStage + slot * C::STAGE_BYTES);
#pragma unroll
            for (int ks = 0; ks < C::VROWS / 16; ++ks) {
              const int key_local = vs * C::VROWS + ks * 16;
              mma_ts(tmem + C::TMEM_O, pcol + key_local / 2,
                     smem_desc_sw128(v_base + ks * 2048, C::V_ATOM_BYTES, 1024), IDESC_O, (j | vs | ks) != 0);
            }
            mma_commit(&empty[slot]);
          }
          mma_commit(bar_o);
          return true;
        };
        for (int j = 0; j < n && ok; ++j) {
          ok = mma_s(j);
          if (ok && j >= 1) ok = mma_o(j - 1);
        }
        if (ok) ok = mma_o(n - 1);
        gs += n;
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
        // let every MMA already issued finish before TMEM is released
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = g.scale_log2;
    using T = typename E::T;
    int gs = 0;  // steps (= P V MMAs) of earlier items
    bool ok = true;
    for (int idx = blockIdx.x; idx < total && ok; idx += gridDim.x) {
      FwdItem t;
      if (!fwd_item<DQK, DV>(p, idx, t)) continue;
      const int n_tiles = t.n;
      const int i = t.q0 + r;
      const int lo_i = t.kr.lo(i), hi_i = t.kr.hi(i);
      const int lo_last = t.kr.lo(t.q_last), hi_first = t.kr.hi(t.q0);
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < n_tiles; ++j) {
        const int sj = gs + j;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar_s[sj & 1], (sj >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t scol = lane_base + C::TMEM_S + (sj & 1) * 128;
        float s[128];
        float mt;  // the tile's row max (the loads return it for an unmasked tile)
        {
          uint32_t u0[32], u1[32], u2[32], u3[32];
          float x0, x1, x2, x3;
          tmem_ld32_max(scol, u0, x0);
          tmem_ld32_max(scol + 32, u1, x1);
          tmem_ld32_max(scol + 64, u2, x2);
          tmem_ld32_max(scol + 96, u3, x3);
          tmem_wait_ld();
          reg_fence(u0);
          reg_fence(u1);
          reg_fence(u2);
          reg_fence(u3);
          asm volatile("" : "+f"(x0), "+f"(x1), "+f"(x2), "+f"(x3));
          mt = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            s[c] = __uint_as_float(u0[c]);
            s[32 + c] = __uint_as_float(u1[c]);
            s[64 + c] = __uint_as_float(u2[c]);
            s[96 + c] = __uint_as_float(u3[c]);
          }
        }
        const int kb = (t.t_lo + j) * C::BN;
        if (!(lo_last <= kb && hi_first >= kb + C::BN)) {  // edge tile (uniform branch)
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = in_range(kb + c, lo_i, hi_i) ? s[c] : -INFINITY;
          float mc[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int c = 4; c < 128; ++c) mc[c & 3] = fmaxf(mc[c & 3], s[c]);
          mt = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
        }
        const float m_new = fmaxf(m_used, mt);
        bool need = false;
        float f = 1.f;
        if (m_used == -INFINITY) {
          m_used = m_new;  // nothing accumulated yet for this row
        } else if ((m_new - m_used) * sl2 > 8.f) {
          need = true;
          f = ex2((m_used - m_new) * sl2);
          m_used = m_new;
        }
        const float mb = (m_used == -INFINITY) ? 0.f : m_used * sl2;
        float rs = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = ex2(fmaf(s[half * 64 + 2 * c], sl2, -mb));
            const float p1 = ex2(fmaf(s[half * 64 + 2 * c + 1], sl2, -mb));
            rs += p0 + p1;
            pk[c] = E::pack(p0, p1);
          }
          tmem_st32(scol + half * 32, pk);
        }
        l = l * f + rs;
        if (j >= 1) {
          // PV_{j-1} must be complete before O is touched (and before P_j is
          // released, which keeps this wait in step with every completion).
          if (!__all_sync(0xffffffffu, mbar_wait(bar_o, (sj - 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
              uint32_t u[32];
              tmem_ld32(lane_base + C::TMEM_O + c * 32, u);
              tmem_wait_ld();
              reg_fence(u);
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * f);
              tmem_st32(lane_base + C::TMEM_O + c * 32, u);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p[sj & 1]);
      }
      if (!ok) break;
      if (n_tiles > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar_o, (gs + n_tiles - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const bool valid = i < t.si.lq;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      T* orow = reinterpret_cast<T*>(p.o) + ((int64_t)(t.si.qrow0 + i) * g.nh_q + t.qhead) * g.dv + t.split * DV;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t packed[16];
        if (n_tiles > 0) {
          uint32_t u[32];
          tmem_ld32(lane_base + C::TMEM_O + c * 32, u);
          tmem_wait_ld();
          reg_fence(u);
          if (c == DV / 32 - 1) {  // every column of O is read: the next item's P V may overwrite it
            tc_fence_before();
            mbar_arrive(o_free);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e)
            packed[e] = E::pack(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) packed[e] = 0u;
        }
        if (valid && SDPA_ADDR_OK(g.chk, orow + c * 32, 64)) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
        }
      }
      float* lse_at = p.lse + (int64_t)(t.si.qrow0 + i) * g.nh_q + t.qhead;
      if (valid && t.split == 0 && SDPA_ADDR_OK(g.chk, lse_at, 4))
        *lse_at = l > 0.f ? m_used * g.scale + logf(l) : -INFINITY;
      gs += n_tiles;
    }
    if (!ok) {
      *abort_flag = 1;
      record_error(p.err, SDPA_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// head_dim 128: a persistent kernel, one CTA per SM running two independent
// query-tile pipelines (384 threads launched at 168 registers, ~195 KB of
// shared memory, all 512 TMEM columns: pipeline X has O at [256X, 256X+128)
// and S/P at [256X+128, 256X+256)). The two softmax warpgroups take 192
// registers a thread and the producer/MMA warpgroup keeps 120
// (2 x 192 + 120 = 3 x 168: both the block's registers and each SM
// sub-partition's, which hosts one warp of every warpgroup). Each pipeline takes query tiles,
// heaviest first, from an atomic ticket counter; TMEM allocation and barrier
// set-up are paid once per CTA, a tile's Q is loaded as soon as the previous
// tile's last S has been issued, and the next tile's first S runs while the
// softmax warps write the current tile's output.
// Within a pipeline a tile runs S_j -> softmax_j -> PV_j in turn (one S
// buffer). The single MMA issuer serves the two pipelines strictly in turn
// (PV_A, S_A, PV_B, S_B, ...), which keeps them half a period apart: one
// pipeline's softmax runs while the tensor pipe works on the other's MMAs.
// (Two separate CTAs per SM, with nothing to order them, drift into step and
// then contend for the same units.)
// Roles: warps 0-3 / 4-7 softmax + epilogue of pipeline 0 / 1 (one thread
// per query row), warps 8 / 9 TMA producer and scheduler of pipeline 0 / 1,
// warp 10 TMEM allocator + MMA issuer, warp 11 only completes the third
// warpgroup. A producer publishes each tile through
// a two-entry queue in shared memory; every barrier phase counts across
// tiles. The softmax makes one pass over S in TMEM per key tile (a second one
// only when a row's max moves).
// One pass of the head_dim 128 softmax over the 128 scores of a row held in
// TMEM: t = S*scale*log2e - mb, P = exp2(t) packed to 16-bit pairs (zero
// where masked), the row sum of P and the largest t among allowed keys.
template <bool MASK, class E>
__device__ __forceinline__ void p_pass(uint32_t scol, float sl2, float mb, int kb, int lo, int hi,
                                       uint32_t (&pk)[64], float& rs, float& tmax) {
  const float2 sc = make_float2(sl2, sl2), nm = make_float2(-mb, -mb);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t u[32];
    float cmax = 0.f;
    if (MASK)
      tmem_ld32(scol + c * 32, u);
    else
      tmem_ld32_max(scol + c * 32, u, cmax);
    tmem_wait_ld();
    reg_fence(u);
    if (!MASK) {
      // the load returned the chunk's max score; the rounding of the exponent
      // being monotone, fma(max, scale*log2e, -mb) is the chunk's largest one
      asm volatile("" : "+f"(cmax));
      tmax = fmaxf(tmax, __fmaf_rn(cmax, sl2, -mb));
    }
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float2 t = ffma2(make_float2(__uint_as_float(u[e]), __uint_as_float(u[e + 1])), sc, nm);
      if (MASK) {
        const int key = kb + c * 32 + e;
        t.x = in_range(key, lo, hi) ? t.x : -INFINITY;
        t.y = in_range(key + 1, lo, hi) ? t.y : -INFINITY;
        tmax = fmaxf(tmax, fmaxf(t.x, t.y));
      }
      const float2 p = make_float2(ex2(t.x), ex2(t.y));
      pk[c * 16 + e / 2] = E::pack(p.x, p.y);
      acc = fadd2(acc, p);
    }
  }
  rs = acc.x + acc.y;
}

struct Fwd2Cfg {
  static constexpr int Q_BYTES = 32768;
  static constexpr int STAGE_BYTES = 32768;
  static constexpr int NSTAGES = 2;
  static constexpr int PIPE_BYTES = Q_BYTES + NSTAGES * STAGE_BYTES;  // per pipeline, 1024-aligned
  static constexpr int PIPE_BARS = 16;                                // mbarriers + queue per pipeline (8 bytes each)
  static constexpr int STG_BYTES = 8 * 2048;  // per softmax warp: 32 rows x 64 bytes of output
  static constexpr int SMEM_BYTES = 1024 + 2 * PIPE_BYTES + 2 * PIPE_BARS * 8 + 32 + STG_BYTES;
  static constexpr uint32_t TMEM_O = 0, TMEM_S = 128, TMEM_PIPE = 256;
  static constexpr int THREADS = 384;
  static constexpr int REGS_SOFTMAX = 192, REGS_OTHER = 120;
  static_assert(2 * REGS_SOFTMAX + REGS_OTHER <= 3 * 168, "register split");
};

// Shared-memory objects of one pipeline.
struct Pipe128 {
  uint8_t* sQ;
  uint8_t* sStage;
  uint64_t* full;         // [NSTAGES]
  uint64_t* empty;        // [NSTAGES]
  uint64_t* bar_q;        // Q of a tile landed
  uint64_t* bar_s;        // S_j ready
  uint64_t* bar_p;        // P_j written (and O rescaled)
  uint64_t* bar_o;        // last PV of a tile done
  uint64_t* q_free;       // every S of a tile done: Q may be replaced
  uint64_t* o_free;       // the epilogue has read O
  uint64_t* sched_full;   // [2] a tile published
  uint64_t* sched_empty;  // [2] its entry read by the MMA issuer and the softmax warps
  int* sched;             // [2] ticket, or -1 when the work is out
};

__device__ __forceinline__ Pipe128 pipe_at(uint8_t* smem, int x) {
  using C = Fwd2Cfg;
  Pipe128 P;
  P.sQ = smem + x * C::PIPE_BYTES;
  P.sStage = P.sQ + C::Q_BYTES;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + 2 * C::PIPE_BYTES) + x * C::PIPE_BARS;
  P.full = b;
  P.empty = b + C::NSTAGES;
  P.bar_q = b + 2 * C::NSTAGES;
  P.bar_s = P.bar_q + 1;
  P.bar_p = P.bar_q + 2;
  P.bar_o = P.bar_q + 3;
  P.q_free = P.bar_q + 4;
  P.o_free = P.bar_q + 5;
  P.sched_full = P.bar_q + 6;
  P.sched_empty = P.bar_q + 8;
  P.sched = reinterpret_cast<int*>(P.bar_q + 10);
  return P;
}

// A query tile of the ticket order (heaviest first: the last query tiles of
// every sequence come first) and the keys it sees.
struct Tile128 {
  int h, b, q0, q_last, t_lo, n;
  SeqInfo si;
  KeyRange kr;
};

__device__ __forceinline__ bool decode_tile(const FwdParams& p, int idx, Tile128& t) {
  const Geom& g = p.g;
  t.h = idx % g.hq;
  idx /= g.hq;
  t.b = idx % g.batch;
  idx /= g.batch;
  t.q0 = (p.n_q_tiles - 1 - idx) * 128;
  t.si = seq_info(g, t.b);
  if (t.q0 >= t.si.lq) return false;
  t.kr = key_range(g, t.si.lq, t.si.lk);
  t.q_last = min(t.q0 + 127, t.si.lq - 1);
  const int lo = t.kr.lo(t.q0), hi = t.kr.hi(t.q_last);
  t.t_lo = lo / 128;
  t.n = hi > lo ? (hi + 127) / 128 - t.t_lo : 0;
  return true;
}

template <bool BF16>
__global__ void __launch_bounds__(Fwd2Cfg::THREADS, 1)
    fwd128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using C = Fwd2Cfg;
  using E = Elem<BF16>;
  const Geom& g = p.g;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar_drain = reinterpret_cast<uint64_t*>(smem + 2 * C::PIPE_BYTES) + 2 * C::PIPE_BARS;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  uint8_t* stg = reinterpret_cast<uint8_t*>(bar_drain) + 32;  // [8 softmax warps][2 KB] output staging
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      const Pipe128 P = pipe_at(smem, x);
      for (int i = 0; i < C::NSTAGES; ++i) {
        mbar_init(&P.full[i], 1);
        mbar_init(&P.empty[i], 1);
      }
      mbar_init(P.bar_q, 1);
      mbar_init(P.bar_s, 1);
      mbar_init(P.bar_p, 128);
      mbar_init(P.bar_o, 1);
      mbar_init(P.q_free, 1);
      mbar_init(P.o_free, 128);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&P.sched_full[i], 1);
        mbar_init(&P.sched_empty[i], 129);
      }
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 10) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp >= 8) {
    regs_dec<C::REGS_OTHER>();
    if (warp == 8 || warp == 9) {
    // ------------------------------------------------------------ scheduler + producer of pipeline warp - 8
    if (elect_one()) {
      const Pipe128 P = pipe_at(smem, warp - 8);
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int c = 0, nq = 0, w = 0;
      bool ok = true;
      // the next ticket (a counter the address check rejects hands out none)
      auto take = [&]() { return SDPA_ADDR_OK(g.chk, p.tile_counter, 4) ? atomicAdd(p.tile_counter, 1) : p.total_tiles; };
      int ticket = take();
      while (true) {
        Tile128 t;
        while (ticket < p.total_tiles && !decode_tile(p, ticket, t)) ticket = take();
        const int item = ticket < p.total_tiles ? ticket : -1;
        const int e = w & 1;
        if (!mbar_wait(&P.sched_empty[e], ((w >> 1) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        P.sched[e] = item;
        mbar_arrive(&P.sched_full[e]);
        ++w;
        if (item < 0) break;
        ticket = take();  // in flight while this tile's loads are issued
        if (t.n == 0) continue;
        if (nq > 0 && !mbar_wait(P.q_free, (nq - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int qhead = t.si.qhead0 + t.h;
        const int khead = t.si.khead0 + t.h / (g.hq / g.hkv);
        mbar_arrive_expect_tx(P.bar_q, C::Q_BYTES);
        tma_load_3d(&tmQ, P.bar_q, P.sQ, 0, qhead, t.si.qrow0 + t.q0);
        tma_load_3d(&tmQ, P.bar_q, P.sQ + 16384, 64, qhead, t.si.qrow0 + t.q0);
        ++nq;
        for (int j = 0; j < t.n && ok; ++j) {
          const int key0 = t.si.krow0 + (t.t_lo + j) * 128;
          for (int kv = 0; kv < 2; ++kv, ++c) {
            const int slot = c % C::NSTAGES;
            if (!mbar_wait(&P.empty[slot], ((c / C::NSTAGES) & 1) ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&P.full[slot], C::STAGE_BYTES);
            const CUtensorMap* m = kv ? &tmV : &tmK;
            uint8_t* dst = P.sStage + slot * C::STAGE_BYTES;
            tma_load_3d(m, &P.full[slot], dst, 0, khead, key0);
            tma_load_3d(m, &P.full[slot], dst + 16384, 64, khead, key0);
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
      const int first = c > C::NSTAGES ? c - C::NSTAGES : 0;
      for (int k = first; k < c; ++k) mbar_wait_drain(&P.full[k % C::NSTAGES], (k / C::NSTAGES) & 1);
      if (nq > 0) mbar_wait_drain(P.bar_q, (nq - 1) & 1);
    }
    } else if (warp == 10) {
    // ------------------------------------------------------------ MMA issuer for both pipelines
    if (elect_one()) {
      constexpr uint32_t IDESC_S = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t IDESC_O = idesc_f16(128, 128, BF16, false, true);
      struct State {
        int w, c, nq, tiles, no, n, j;
        bool done;
      };
      State st[2];
      for (int x = 0; x < 2; ++x) st[x] = State{0, 0, 0, 0, 0, 0, 0, false};
      bool ok = true;
      // next tile with keys of pipeline x (false: its work is out, or a wait failed)
      auto next_item = [&](int x) -> bool {
        const Pipe128 P = pipe_at(smem, x);
        State& m = st[x];
        while (true) {
          const int e = m.w & 1;
          if (!mbar_wait(&P.sched_full[e], (m.w >> 1) & 1, abort_flag)) {
            ok = false;
            return false;
          }
          const int item = *reinterpret_cast<volatile int*>(&P.sched[e]);
          mbar_arrive(&P.sched_empty[e]);
          ++m.w;
          if (item < 0) {
            m.done = true;
            return false;
          }
          Tile128 t;
          decode_tile(p, item, t);
          if (t.n == 0) continue;
          if (!mbar_wait(P.bar_q, m.nq & 1, abort_flag)) {
            ok = false;
            return false;
          }
          ++m.nq;
          tc_fence_after();
          m.n = t.n;
          m.j = 0;
          return true;
        }
      };
      // S_j = Q K_j^T of pipeline x (its previous PV has been issued, so P_{j-1} is consumed first)
      auto issue_s = [&](int x) -> bool {
        const Pipe128 P = pipe_at(smem, x);
        State& m = st[x];
        const int slot = m.c % C::NSTAGES;
        if (!mbar_wait(&P.full[slot], (m.c / C::NSTAGES) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t q_base = smem_u32(P.sQ), base = smem_u32(P.sStage + slot * C::STAGE_BYTES);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          mma_ss(tmem + x * C::TMEM_PIPE + C::TMEM_S, smem_desc_sw128(q_base + off, 16, 1024),
                 smem_desc_sw128(base + off, 16, 1024), IDESC_S, ks != 0);
        }
        mma_commit(&P.empty[slot]);
        if (m.j == m.n - 1) mma_commit(P.q_free);
        mma_commit(P.bar_s);
        ++m.c;
        return true;
      };
      // O += P_j V_j of pipeline x; the first PV of a tile overwrites O, which
      // the previous tile's epilogue must have read
      auto issue_pv = [&](int x) -> bool {
        const Pipe128 P = pipe_at(smem, x);
        State& m = st[x];
        if (m.j == 0 && m.no > 0 && !mbar_wait(P.o_free, (m.no - 1) & 1, abort_flag)) return false;
        if (!mbar_wait(P.bar_p, m.tiles & 1, abort_flag)) return false;
        ++m.tiles;
        const int slot = m.c % C::NSTAGES;
        if (!mbar_wait(&P.full[slot], (m.c / C::NSTAGES) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t base = smem_u32(P.sStage + slot * C::STAGE_BYTES);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tmem + x * C::TMEM_PIPE + C::TMEM_O, tmem + x * C::TMEM_PIPE + C::TMEM_S + ks * 8,
                 smem_desc_sw128(base + ks * 2048, 16384, 1024), IDESC_O, (m.j | ks) != 0);
        mma_commit(&P.empty[slot]);
        ++m.c;
        return true;
      };
      for (int x = 0; x < 2 && ok; ++x)
        if (next_item(x) && !issue_s(x)) ok = false;
      while (ok && !(st[0].done && st[1].done)) {
        for (int x = 0; x < 2 && ok; ++x) {
          State& m = st[x];
          if (m.done) continue;
          if (!issue_pv(x)) {
            ok = false;
            break;
          }
          if (m.j == m.n - 1) {
            mma_commit(pipe_at(smem, x).bar_o);
            ++m.no;
            if (!next_item(x)) continue;  // out of work (or ok cleared)
          } else {
            ++m.j;
          }
          if (!issue_s(x)) ok = false;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    }
    }
  } else {
    regs_inc<C::REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax + epilogue of pipeline warp / 4
    const int x = warp >> 2;
    const Pipe128 P = pipe_at(smem, x);
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + x * C::TMEM_PIPE + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t scol = lane_base + C::TMEM_S;
    const float sl2 = g.scale_log2;
    int w = 0, tiles = 0, no = 0;
    bool ok = true;
    while (ok) {
      const int e = w & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&P.sched_full[e], (w >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      const int item = *reinterpret_cast<volatile int*>(&P.sched[e]);
      mbar_arrive(&P.sched_empty[e]);
      ++w;
      if (item < 0) break;
      int lo_i, hi_i, lo_last, hi_first, t_lo, n;
      bool valid;
      typename E::T* orow;  // this row's output and LSE, kept for the epilogue
      float* lse_at;
      {
        Tile128 t;
        decode_tile(p, item, t);
        const int i = t.q0 + r;
        lo_i = t.kr.lo(i);
        hi_i = t.kr.hi(i);
        lo_last = t.kr.lo(t.q_last);
        hi_first = t.kr.hi(t.q0);
        t_lo = t.t_lo;
        n = t.n;
        valid = i < t.si.lq;
        const int qhead = t.si.qhead0 + t.h;
        orow = reinterpret_cast<typename E::T*>(p.o) + ((int64_t)(t.si.qrow0 + i) * g.nh_q + qhead) * 128;
        lse_at = p.lse + (int64_t)(t.si.qrow0 + i) * g.nh_q + qhead;
      }
      float mbs = -INFINITY, l = 0.f;  // running max of S*scale*log2e, and the row sum
      for (int j = 0; j < n; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(P.bar_s, tiles & 1, abort_flag))) {
          ok = false;
          break;
        }
        ++tiles;
        tc_fence_after();
        const int kb = (t_lo + j) * 128;
        const bool interior = lo_last <= kb && hi_first >= kb + 128;
        // One pass: P against the running max m (P = exp2(S*scale*log2e - m)),
        // keeping the largest exponent t. While t <= 8 every P is <= 256 and
        // m can stay as it is. A row whose scores jumped higher (or that sees
        // its first allowed key) is recomputed against its new max (S is still
        // intact in TMEM: P is only written back after the check), and O and l
        // are rescaled by exp2(-t).
        const float mb = (mbs == -INFINITY) ? 0.f : mbs;
        float rs = 0.f, tmax = -INFINITY;
        uint32_t pk[64];
        if (interior)
          p_pass<false, E>(scol, sl2, mb, kb, lo_i, hi_i, pk, rs, tmax);
        else
          p_pass<true, E>(scol, sl2, mb, kb, lo_i, hi_i, pk, rs, tmax);
        // A row's first allowed keys always take the second pass, against its
        // exact max: its largest P is then exactly 1, so the rounding of the
        // dominant P cannot bias O against the LSE.
        const bool redo = tmax > 8.f || (mbs == -INFINITY && tmax > -INFINITY);
        float f = 1.f;
        if (__any_sync(0xffffffffu, redo)) {
          // the whole warp repeats the pass (TMEM loads are warp-wide); rows
          // that keep their max recompute bit-identical values
          const float mb2 = redo ? mb + tmax : mb;
          float t2 = -INFINITY;
          if (interior)
            p_pass<false, E>(scol, sl2, mb2, kb, lo_i, hi_i, pk, rs, t2);
          else
            p_pass<true, E>(scol, sl2, mb2, kb, lo_i, hi_i, pk, rs, t2);
        }
        if (redo) {
          f = mbs == -INFINITY ? 0.f : ex2(-tmax);
          mbs = mb + tmax;
        }
        l = l * f + rs;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t q16[16];
#pragma unroll
          for (int k2 = 0; k2 < 16; ++k2) q16[k2] = pk[cc * 16 + k2];
          tmem_st16(scol + cc * 16, q16);
        }
        // PV_{j-1} completed before S_j was computed (single S buffer), so O
        // can be rescaled here without waiting.
        if (__any_sync(0xffffffffu, f != 1.f) && j > 0) {
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t u[32];
            tmem_ld32(lane_base + C::TMEM_O + cc * 32, u);
            tmem_wait_ld();
            reg_fence(u);
#pragma unroll
            for (int k2 = 0; k2 < 32; ++k2) u[k2] = __float_as_uint(__uint_as_float(u[k2]) * f);
            tmem_st32(lane_base + C::TMEM_O + cc * 32, u);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(P.bar_p);
      }
      if (!ok) break;
      // epilogue: O / l, 32 columns at a time; O is free for the next tile's
      // first PV once the last chunk has been read
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (n > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(P.bar_o, no & 1, abort_flag))) {
          ok = false;
          break;
        }
        ++no;
        tc_fence_after();
      }
      // 32 columns (64 bytes of a row) at a time, staged in shared memory so
      // that each store writes eight rows' 64 contiguous bytes
      uint8_t* wst = stg + warp * 2048;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t packed[16];
        if (n > 0) {
          uint32_t u[32];
          tmem_ld32(lane_base + C::TMEM_O + cc * 32, u);
          tmem_wait_ld();
          reg_fence(u);
          if (cc == 3) {
            tc_fence_before();
            mbar_arrive(P.o_free);
          }
#pragma unroll
          for (int k2 = 0; k2 < 16; ++k2)
            packed[k2] = E::pack(__uint_as_float(u[2 * k2]) * inv, __uint_as_float(u[2 * k2 + 1]) * inv);
        } else {
#pragma unroll
          for (int k2 = 0; k2 < 16; ++k2) packed[k2] = 0u;
        }
        // segment k2 of row `lane` at position k2 ^ (lane % 4): four wavefronts a store
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2)
          *reinterpret_cast<uint4*>(wst + lane * 64 + ((k2 ^ (lane & 3)) << 4)) =
              make_uint4(packed[4 * k2], packed[4 * k2 + 1], packed[4 * k2 + 2], packed[4 * k2 + 3]);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = k * 8 + (lane >> 2), seg = lane & 3;  // row of the warp, 16-byte segment
          const uint4 v4 = *reinterpret_cast<const uint4*>(wst + rr * 64 + ((seg ^ (rr & 3)) << 4));
          typename E::T* dst = reinterpret_cast<typename E::T*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(orow), rr));
          const bool vr = __shfl_sync(0xffffffffu, valid ? 1 : 0, rr) != 0;
          if (vr && SDPA_ADDR_OK(g.chk, dst + cc * 32 + seg * 8, 16))
            *reinterpret_cast<uint4*>(dst + cc * 32 + seg * 8) = v4;
        }
        __syncwarp();
      }
      if (valid && SDPA_ADDR_OK(g.chk, lse_at, 4)) *lse_at = l > 0.f ? mbs * 0.6931471805599453f + logf(l) : -INFINITY;
    }
    if (!ok) {
      *abort_flag = 1;
      record_error(p.err, SDPA_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BF16>
static int launch_fwd128(const FwdLaunch& L) {
  auto kern = fwd128_kernel<BF16>;
  if (const int rc = set_kernel_smem(reinterpret_cast<const void*>(kern), Fwd2Cfg::SMEM_BYTES, 100)) return rc;
  const long long tiles = (long long)L.p.n_q_tiles * L.p.g.hq * L.p.g.batch;
  if (tiles <= 0) return SDPA_OK;
  if (tiles > 0x7fffffffLL - 4096) return SDPA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDPA_ERR_CUDA;
  FwdParams p = L.p;
  p.total_tiles = (int)tiles;
  long long grid = std::min<long long>((tiles + 1) / 2, sms);
  if (debug_max_ctas() > 0) grid = std::min<long long>(grid, debug_max_ctas());  // tickets cover every tile
  if (cudaMemsetAsync(p.tile_counter, 0, sizeof(int), L.stream) != cudaSuccess) return SDPA_ERR_CUDA;
  kern<<<(unsigned)grid, Fwd2Cfg::THREADS, Fwd2Cfg::SMEM_BYTES, L.stream>>>(L.tmQ, L.tmK, L.tmV, p);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

template <int DQK, int DV, bool BF16>
static int launch_fwd_t(const FwdLaunch& L) {
  using C = FwdCfg<DQK, DV>;
  auto kern = fwd_kernel<DQK, DV, BF16>;
  if (const int rc = set_kernel_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, -1)) return rc;
  const long long items = (long long)L.p.n_q_tiles * L.p.g.hq * L.p.g.batch * L.p.dv_splits;
  if (items <= 0) return SDPA_OK;
  if (items > 0x7fffffffLL - 4096) return SDPA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDPA_ERR_CUDA;
  FwdParams p = L.p;
  p.total_tiles = (int)items;
  long long grid = std::min<long long>(items, sms);
  if (debug_max_ctas() > 0) grid = std::min<long long>(grid, debug_max_ctas());  // the CTAs stride over every item
  kern<<<(unsigned)grid, 256, C::SMEM_BYTES, L.stream>>>(L.tmQ, L.tmK, L.tmV, p);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

int launch_fwd(const FwdLaunch& L, int head_dim, int head_dim_v, bool bf16) {
  if (head_dim == 192 && head_dim_v == 128)
    return bf16 ? launch_fwd_t<192, 128, true>(L) : launch_fwd_t<192, 128, false>(L);
  if (head_dim != head_dim_v) return SDPA_ERR_UNSUPPORTED;
  if (head_dim == 128) return bf16 ? launch_fwd128<true>(L) : launch_fwd128<false>(L);
  if (head_dim == 256) return bf16 ? launch_fwd_t<256, 256, true>(L) : launch_fwd_t<256, 256, false>(L);
  if (head_dim == 512) return bf16 ? launch_fwd_t<512, 256, true>(L) : launch_fwd_t<512, 256, false>(L);
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace sdpa
