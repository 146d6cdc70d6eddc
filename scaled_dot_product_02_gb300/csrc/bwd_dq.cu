// bwd_dq.cu -- deterministic dQ for head_dim 128 (no atomics).
//
// The default head_dim 128 backward accumulates dQ with fp32 reductions from
// every key tile's CTA, so its dQ is not bitwise reproducible run to run.
// The deterministic backward (TransformerEngine PR #3527 records
// deterministic execution as unavailable for the prior art's kernels) runs
// the dK/dV kernel without its dQ part and this kernel after it: one CTA per
// (128-query tile, q head, batch) walks the key tiles the tile can see in a
// fixed order and accumulates dQ in TMEM, recomputing per key tile
//   S  = Q K^T, dP = dO V^T             (SS, fp32 in TMEM)
//   P  = exp2(S*scale*log2e - LSE*log2e) (masked),  dS = P * (dP - delta)
//   dQ += dS K                           (TS, dS read as 16-bit from TMEM)
// and writes dQ * scale once. Two of its three GEMMs repeat work the dK/dV
// kernel does; that is the price of a fixed summation order.
//
// Roles (192 threads): warps 0-3 one thread per query row (P, dS, and the dQ
// epilogue), warp 4 TMA producer (Q and dO once, then K_j and V_j through a
// ring of four 32 KB stages), warp 5 TMEM allocator and MMA issuer.
// TMEM: S [0,128) (dS packed into its first 64 columns), dP [128,256),
// dQ [256,384).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

struct DqCfg {
  static constexpr int Q_BYTES = 32768;      // 128 rows x 128 columns, two 64-column atoms
  static constexpr int STAGE_BYTES = 32768;  // one K or V tile
  static constexpr int NSTAGES = 4;
  static constexpr int NBARS = 2 * NSTAGES + 5;
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + NSTAGES * STAGE_BYTES + NBARS * 8 + 16;
  static constexpr uint32_t TMEM_S = 0, TMEM_DP = 128, TMEM_DQ = 256;
};

// dS for 32 keys of one query row, packed to 16-bit pairs.
template <bool MASK, class E>
__device__ __forceinline__ void ds_cols(const uint32_t (&us)[32], const uint32_t (&ud)[32], float sl2, float nl2,
                                        float dl, int key0, int lo, int hi, uint32_t (&pd)[16]) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float p0 = ex2(fmaf(__uint_as_float(us[c]), sl2, nl2));
    float p1 = ex2(fmaf(__uint_as_float(us[c + 1]), sl2, nl2));
    if (MASK) {
      p0 = in_range(key0 + c, lo, hi) ? p0 : 0.f;
      p1 = in_range(key0 + c + 1, lo, hi) ? p1 : 0.f;
    }
    pd[c / 2] = E::pack(p0 * (__uint_as_float(ud[c]) - dl), p1 * (__uint_as_float(ud[c + 1]) - dl));
  }
}

}  // namespace

template <bool BF16>
__global__ void __launch_bounds__(192, 1)
    dq128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ DqParams p) {
  using C = DqCfg;
  using E = Elem<BF16>;
  const Geom& g = p.g;
  int idx = blockIdx.x + p.item_offset;
  const int h = idx % g.hq;
  idx /= g.hq;
  const int b = idx % g.batch;
  idx /= g.batch;
  const int qt = p.n_q_tiles - 1 - idx;  // heaviest query tiles first
  const SeqInfo si = seq_info(g, b);
  const int q0 = qt * 128;
  if (q0 >= si.lq) return;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;
  const KeyRange kr = key_range(g, si.lq, si.lk);
  const int q_last = min(q0 + 127, si.lq - 1);
  const int kv_lo = kr.lo(q0), kv_hi = kr.hi(q_last);
  const int t_lo = kv_lo / 128;
  const int n_tiles = (kv_hi > kv_lo) ? (kv_hi + 127) / 128 - t_lo : 0;
  const int qhead = si.qhead0 + h;
  const int khead = si.khead0 + h / (g.hq / g.hkv);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::Q_BYTES;
  uint8_t* sStage = smem + 2 * C::Q_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + C::NSTAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::NSTAGES;
  uint64_t* bar_q = empty + C::NSTAGES;  // Q and dO landed
  uint64_t* bar_sdp = bar_q + 1;         // S_j and dP_j ready
  uint64_t* bar_ds = bar_sdp + 1;        // dS_j written to TMEM
  uint64_t* bar_dq = bar_ds + 1;         // the last dQ MMA done
  uint64_t* bar_drain = bar_dq + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSTAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(bar_q, 1);
    mbar_init(bar_sdp, 1);
    mbar_init(bar_ds, 128);
    mbar_init(bar_dq, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 4) {
    // ------------------------------------------------------------ producer: Q, dO, then K_0, V_0, K_1, V_1, ...
    if (elect_one() && n_tiles > 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(bar_q, 2 * C::Q_BYTES);
      for (int a = 0; a < 2; ++a) {
        tma_load_3d(&tmQ, bar_q, sQ + a * 16384, a * 64, qhead, si.qrow0 + q0);
        tma_load_3d(&tmDO, bar_q, sDO + a * 16384, a * 64, qhead, si.qrow0 + q0);
      }
      int c = 0;
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int key0 = si.krow0 + (t_lo + j) * 128;
        for (int kv = 0; kv < 2; ++kv, ++c) {
          const int slot = c % C::NSTAGES;
          if (!mbar_wait(&empty[slot], ((c / C::NSTAGES) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], C::STAGE_BYTES);
          const CUtensorMap* m = kv ? &tmV : &tmK;
          uint8_t* dst = sStage + slot * C::STAGE_BYTES;
          tma_load_3d(m, &full[slot], dst, 0, khead, key0);
          tma_load_3d(m, &full[slot], dst + 16384, 64, khead, key0);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
      const int first = c > C::NSTAGES ? c - C::NSTAGES : 0;
      for (int k = first; k < c; ++k) mbar_wait_drain(&full[k % C::NSTAGES], (k / C::NSTAGES) & 1);
      mbar_wait_drain(bar_q, 0);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one() && n_tiles > 0) {
      constexpr uint32_t ID_SS = idesc_f16(128, 128, BF16, false, false);  // S, dP: both K-major
      constexpr uint32_t ID_DQ = idesc_f16(128, 128, BF16, false, true);   // dQ: B = K tile, N (= D) major
      bool ok = mbar_wait(bar_q, 0, abort_flag);
      tc_fence_after();
      const uint32_t q_base = smem_u32(sQ), do_base = smem_u32(sDO);
      int c = 0;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int sk = c % C::NSTAGES, sv = (c + 1) % C::NSTAGES;
        // S_j = Q K_j^T (overwrites dS_{j-1}, which the dQ MMA issued before it has read)
        if (!mbar_wait(&full[sk], (c / C::NSTAGES) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = smem_u32(sStage + sk * C::STAGE_BYTES);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          mma_ss(tmem + C::TMEM_S, smem_desc_sw128(q_base + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024), ID_SS,
                 ks != 0);
        }
        // dP_j = dO V_j^T
        if (!mbar_wait(&full[sv], ((c + 1) / C::NSTAGES) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vb = smem_u32(sStage + sv * C::STAGE_BYTES);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          mma_ss(tmem + C::TMEM_DP, smem_desc_sw128(do_base + off, 16, 1024), smem_desc_sw128(vb + off, 16, 1024),
                 ID_SS, ks != 0);
        }
        mma_commit(&empty[sv]);
        mma_commit(bar_sdp);
        // dQ += dS_j K_j
        if (!mbar_wait(bar_ds, j & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tmem + C::TMEM_DQ, tmem + C::TMEM_S + ks * 8, smem_desc_sw128(kb + ks * 2048, 16384, 1024), ID_DQ,
                 (j | ks) != 0);
        mma_commit(&empty[sk]);
        c += 2;
      }
      if (ok) {
        mma_commit(bar_dq);
      } else {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ dS (warps 0-3) and the dQ epilogue
    const int r = warp * 32 + lane;
    const int i = q0 + r;
    const bool valid = i < si.lq;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const long long stat = (long long)qhead * p.stat_rows + si.srow0 + i;
    // rows past the sequence end belong to no query: an empty key range
    const float nl2 = valid && SDPA_ADDR_OK(g.chk, p.nlse2 + stat, 4) ? p.nlse2[stat] : 0.f;
    const float dl = valid && SDPA_ADDR_OK(g.chk, p.delta + stat, 4) ? p.delta[stat] : 0.f;
    const int lo_i = kr.lo(i), hi_i = valid ? kr.hi(i) : lo_i;
    const int lo_last = kr.lo(q_last), hi_first = kr.hi(q0);
    const float sl2 = g.scale_log2;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar_sdp, j & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kb = (t_lo + j) * 128;
      const bool interior = valid && lo_last <= kb && hi_first >= kb + 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t us[32], ud[32], pd[16];
        tmem_ld32(lane_base + C::TMEM_S + cc * 32, us);
        tmem_ld32(lane_base + C::TMEM_DP + cc * 32, ud);
        tmem_wait_ld();
        reg_fence(us);
        reg_fence(ud);
        if (__all_sync(0xffffffffu, interior))
          ds_cols<false, E>(us, ud, sl2, nl2, dl, 0, 0, 0, pd);
        else
          ds_cols<true, E>(us, ud, sl2, nl2, dl, kb + cc * 32, lo_i, hi_i, pd);
        // packed dS of keys 32cc.. goes to columns 16cc.., which hold scores
        // this thread has already read
        tmem_st16(lane_base + C::TMEM_S + cc * 16, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ds);
    }
    if (ok && n_tiles > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dq, 0, abort_flag));
      tc_fence_after();
    }
    if (!ok) {
      *abort_flag = 1;
      record_error(p.err, SDPA_ERR_TIMEOUT);
    } else {
      // every lane takes part in the TMEM loads (warp-wide instructions);
      // only rows inside the sequence are stored
      using T = typename E::T;
      T* row = reinterpret_cast<T*>(p.dq) + ((int64_t)(si.qrow0 + i) * g.nh_q + qhead) * 128;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t packed[16];
        if (n_tiles > 0) {
          uint32_t u[32];
          tmem_ld32(lane_base + C::TMEM_DQ + cc * 32, u);
          tmem_wait_ld();
          reg_fence(u);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            packed[e] = E::pack(__uint_as_float(u[2 * e]) * g.scale, __uint_as_float(u[2 * e + 1]) * g.scale);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) packed[e] = 0u;
        }
        if (valid && SDPA_ADDR_OK(g.chk, row + cc * 32, 64)) {
          uint4* d4 = reinterpret_cast<uint4*>(row + cc * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BF16>
static int launch_dq_t(const DqLaunch& L) {
  auto kern = dq128_kernel<BF16>;
  if (const int rc = set_kernel_smem(reinterpret_cast<const void*>(kern), DqCfg::SMEM_BYTES, -1)) return rc;
  const long long grid = (long long)L.p.n_q_tiles * L.p.g.hq * L.p.g.batch;
  if (grid <= 0) return SDPA_OK;
  if (grid > 0x7fffffffLL) return SDPA_ERR_UNSUPPORTED;
  return launch_in_grids(grid, [&](long long off, long long n) {
    DqParams p = L.p;
    p.item_offset = (int)off;
    kern<<<(unsigned)n, 192, DqCfg::SMEM_BYTES, L.stream>>>(L.tmQ, L.tmDO, L.tmK, L.tmV, p);
    return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
  });
}

int launch_dq128(const DqLaunch& L, bool bf16) { return bf16 ? launch_dq_t<true>(L) : launch_dq_t<false>(L); }

}  // namespace sdpa
