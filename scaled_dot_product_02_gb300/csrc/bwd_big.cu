// bwd_big.cu -- attention backward for head_dim 256 and 512 on sm_103a.
//
// At these head dims the dK and dV accumulators of one 128-key tile need
// 2*D fp32 TMEM columns (512 or 1024) and do not fit next to the score
// tiles, so the backward runs in two phases:
//
// Phase 1, score kernels (one CTA per 128-query tile of one (batch, q head),
// one kernel per head dim, below): S = Q K^T and dP = dO V^T over the full
// head dim for each key tile, P = exp2(S*scale*log2e - LSE*log2e) masked and
// dS = P * (dP - delta) in fp32, P and dS written as 16-bit 128x128 tiles.
//   Each 16-bit tile is stored as the exact shared-memory image a tcgen05 operand
//   wants (two 64-column atoms, 128-byte swizzle), so phase 2 fetches it with
//   one 32 KB bulk copy.
// Phase 2, GEMM kernels (accumulator 128 x 256 fp32 in TMEM, one CTA per
// 256-column slice of the head dim), iterating only over unmasked tiles:
//   MODE_DQ: dQ[q tile]  = scale * sum_t dS(q, t) K(t)
//   MODE_DV: dV[kv tile] = sum_{heads of the group, q tiles} P^T dO
//   MODE_DK: dK[kv tile] = scale * sum dS^T Q
// Every FLOP executed is one the definition counts (10*D per unmasked pair),
// at the cost of 4 bytes of workspace per pair, written once and read back.
//
// Bounded workspace (TransformerEngine PR #3527, "Known limitations": the
// prior art's backward workspace grows from 1.6 GiB at 4k to 74 GiB at 64k
// tokens and caps the context length). The key tiles are processed in chunks
// [chunk_lo, chunk_hi): phase 1 then phase 2 per chunk, so the tile arrays
// hold one chunk at a time, indexed by (batch, head, query tile, slot) with
// slot = key tile - max(first key tile of the query tile, chunk_lo). The host
// sizes the slot count from the mask (a bounded window's span) and from the
// chunk length, never from the whole key range when that would exceed its
// budget. dK and dV of a chunk's key tiles are final after the chunk; dQ of
// a chunk is added (fp32 vector reduce-add, one per element per chunk, the
// chunks ordered by the stream, so the sum is bitwise reproducible) into an
// fp32 accumulator that a last pass scales and converts. With one chunk, dQ
// is written directly.
#include <algorithm>

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr int TILE_BYTES = 128 * 128 * 2;  // one 16-bit 128x128 tile image
constexpr int CHUNK_BYTES = 32768;         // 128 rows x 128 columns of a 16-bit operand

// Bulk store shared -> global (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(gdst)),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}

// Byte offset of 16-byte chunk `k16` (0..15, eight 16-bit values each) of row
// r inside a tile image: two 64-column atoms of [128 rows x 128 bytes], each
// row's chunks permuted by the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_chunk_off(int r, int k16) {
  return (uint32_t)((k16 >> 3) * 16384 + r * 128 + (((k16 & 7) ^ (r & 7)) * 16));
}

// First key tile and number of key tiles that query tile [q0, q0+128) sees.
__device__ __forceinline__ void kv_tiles_of(const KeyRange& kr, int q0, int lq, int& t_lo, int& n) {
  const int q_last = min(q0 + 127, lq - 1);
  const int lo = kr.lo(q0), hi = kr.hi(q_last);
  t_lo = lo / 128;
  n = hi > lo ? (hi + 127) / 128 - t_lo : 0;
}

// Restrict a query tile's key tiles [t_lo, t_lo + n) to this launch's chunk.
__device__ __forceinline__ void chunk_clip(const BigBwdParams& p, int& t_lo, int& n) {
  const int a = max(t_lo, p.chunk_lo), e = min(t_lo + n, p.chunk_hi);
  t_lo = a;
  n = max(0, e - a);
}

__device__ __forceinline__ long long tile_index(const BigBwdParams& p, int b, int h, int qt, int slot) {
  return (((long long)b * p.g.hq + h) * p.n_q_tiles + qt) * p.slots + slot;
}

}  // namespace

// ====================================================================== phase 1
// ---------------------------------------------------------------------- head_dim 256
// Both passes in one kernel. Q and dO of the query tile live in TMEM as the A
// operands of S = Q K^T and dP = dO V^T (columns 0-255), so shared memory is
// left to a deep ring of 16 KB chunks and the staging of the outputs. Q and
// dO arrive through the first eight ring chunks and are copied to TMEM by the
// epilogue threads; K and V follow in the same ring. S (columns 256-383) and
// dP (384-511) are single-buffered but released separately, so S of the next
// key tile is computed while the epilogue waits for dP of this one. Two
// epilogue warpgroups each take 64 keys of a tile: they form P and dS in fp32
// (each rounded once), stage their 64-key atom of both 16-bit tile images and
// write them with bulk copies. Nothing fp32 goes through HBM.
constexpr int SF_CH = 16384;  // ring chunk: 128 rows x 64 columns (one box)
constexpr int SF_NST = 10;
constexpr int SF_STG = 16384;  // one 64-key atom of a tile image
constexpr int SF_NBARS = 2 * SF_NST + 6;
constexpr int SF_SMEM = 1024 + SF_NST * SF_CH + 4 * SF_STG + SF_NBARS * 8 + 16;
constexpr int SF_THREADS = 320;  // producer, MMA, two epilogue warpgroups (warps 2-5, 6-9)
constexpr int SF_TM_Q = 0, SF_TM_DO = 128, SF_TM_S = 256, SF_TM_DP = 384;

template <bool BF16>
__global__ void __launch_bounds__(SF_THREADS, 1)
    score_fused256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                          const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ BigBwdParams p) {
  using E = Elem<BF16>;
  const Geom& g = p.g;
  int idx = blockIdx.x + p.item_offset;
  const int h = idx % g.hq;
  idx /= g.hq;
  const int b = idx % g.batch;
  const int qt = p.n_q_tiles - 1 - idx / g.batch;
  const SeqInfo si = seq_info(g, b);
  const int q0 = qt * 128;
  if (q0 >= si.lq) return;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;
  const KeyRange kr = key_range(g, si.lq, si.lk);
  int t_lo, n;
  kv_tiles_of(kr, q0, si.lq, t_lo, n);
  chunk_clip(p, t_lo, n);
  if (n > p.slots) {
    if (threadIdx.x == 0) record_error(p.err, SDPA_ERR_INVALID_ARG);
    return;
  }
  if (n == 0) return;
  const int qhead = si.qhead0 + h;
  const int khead = si.khead0 + h / (g.hq / g.hkv);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sRing = smem;
  uint8_t* sStg = sRing + SF_NST * SF_CH;  // [group][P, dS] atoms
  uint64_t* full = reinterpret_cast<uint64_t*>(sStg + 4 * SF_STG);
  uint64_t* empty = full + SF_NST;
  uint64_t* bar_qd = empty + SF_NST;  // Q and dO are in TMEM
  uint64_t* bar_s = bar_qd + 1;       // S of a key tile ready
  uint64_t* bar_dp = bar_s + 1;       // dP of a key tile ready
  uint64_t* free_s = bar_dp + 1;      // the epilogue has read S
  uint64_t* free_dp = free_s + 1;     // ... and dP
  uint64_t* bar_drain = free_dp + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SF_NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(bar_qd, 256);
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(free_s, 256);
    mbar_init(free_dp, 256);
    mbar_init(bar_drain, 1);
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

  // ring chunk c: c < 8 are Q (columns 64c..) and dO (64(c-4)..) of the query
  // tile; from c = 8 on, per key tile, K columns 0, 64, 128, 192, then V
  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int total = 8 + 8 * n;
      int c = 0;
      for (; c < total; ++c) {
        const int slot = c % SF_NST;
        if (!mbar_wait(&empty[slot], ((c / SF_NST) & 1) ^ 1, abort_flag)) break;
        uint8_t* dst = sRing + slot * SF_CH;
        mbar_arrive_expect_tx(&full[slot], SF_CH);
        if (c < 8) {
          tma_load_3d(c < 4 ? &tmQ : &tmDO, &full[slot], dst, (c & 3) * 64, qhead, si.qrow0 + q0);
        } else {
          const int t = (c - 8) >> 3, kc = (c - 8) & 7;
          tma_load_3d(kc < 4 ? &tmK : &tmV, &full[slot], dst, (kc & 3) * 64, khead, si.krow0 + (t_lo + t) * 128);
        }
      }
      if (c < total) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
      const int first = c > SF_NST ? c - SF_NST : 0;
      for (int k = first; k < c; ++k) mbar_wait_drain(&full[k % SF_NST], (k / SF_NST) & 1);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t IDESC = idesc_f16(128, 128, BF16, false, false);
      bool ok = mbar_wait(bar_qd, 0, abort_flag);
      tc_fence_after();
      int c = 8;
      for (int t = 0; t < n && ok; ++t) {
        for (int pass = 0; pass < 2 && ok; ++pass) {  // S = Q K^T, then dP = dO V^T
          if (t >= 1 && !mbar_wait(pass == 0 ? free_s : free_dp, (t - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (pass == 0 ? SF_TM_S : SF_TM_DP);
          const uint32_t aa = tmem + (pass == 0 ? SF_TM_Q : SF_TM_DO);
          for (int kc = 0; kc < 4; ++kc, ++c) {
            const int slot = c % SF_NST;
            if (!mbar_wait(&full[slot], (c / SF_NST) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t bb = smem_u32(sRing + slot * SF_CH);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ts(d, aa + kc * 32 + ks * 8, smem_desc_sw128(bb + ks * 32, 16, 1024), IDESC, (kc | ks) != 0);
            mma_commit(&empty[slot]);
          }
          if (ok) mma_commit(pass == 0 ? bar_s : bar_dp);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    }
  } else if (warp >= 2) {
    const int grp = (warp - 2) >> 2;  // 64-key half of each tile; for the TMEM fill, Q (0) or dO (1)
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    const int i = q0 + r;
    const bool valid = i < si.lq;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const bool leader = ((threadIdx.x - 64) & 127) == 0;
    const int bar_id = 1 + grp;
    bool ok = true;
    {
      // row r of Q (group 0) or dO (group 1): ring chunks 4*grp.. -> TMEM, packed pairs along D
      for (int a = 0; a < 4; ++a) {
        const int slot = grp * 4 + a;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], 0, abort_flag)) && ok;
        const uint8_t* row = sRing + slot * SF_CH + r * 128;
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
          v[4 * j] = x.x;
          v[4 * j + 1] = x.y;
          v[4 * j + 2] = x.z;
          v[4 * j + 3] = x.w;
        }
        tmem_st32(lane_base + (grp == 0 ? SF_TM_Q : SF_TM_DO) + a * 32, v);
      }
      tmem_wait_st();
      ok = named_bar_and(bar_id, 128, ok);  // every row of this group has been read out of the ring
      if (ok) {
        if (leader)
          for (int a = 0; a < 4; ++a) mbar_arrive(&empty[grp * 4 + a]);
        tc_fence_before();
        mbar_arrive(bar_qd);
      }
    }
    const long long stat = (long long)qhead * p.stat_rows + si.srow0 + i;
    // rows past the sequence end belong to no query: an empty key range, so
    // their P and dS are exactly zero whatever their scores
    const float nl2 = valid && SDPA_ADDR_OK(g.chk, p.nlse2 + stat, 4) ? p.nlse2[stat] : 0.f;
    const float dl = valid && SDPA_ADDR_OK(g.chk, p.delta + stat, 4) ? p.delta[stat] : 0.f;
    const int lo_i = kr.lo(i), hi_i = valid ? kr.hi(i) : lo_i;
    const float sl2 = g.scale_log2;
    uint8_t* stP = sStg + grp * 2 * SF_STG;
    uint8_t* stD = stP + SF_STG;
    for (int t = 0; t < n && ok; ++t) {
      bool okw = __all_sync(0xffffffffu, mbar_wait(bar_s, t & 1, abort_flag));
      if (leader) bulk_wait_group_read0();  // this group's previous atoms have left the staging
      if (!named_bar_and(bar_id, 128, okw)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kbase = (t_lo + t) * 128 + grp * 64;
      float pv[64];
      {
        uint32_t u[64];
        tmem_ld32(lane_base + SF_TM_S + grp * 64, *reinterpret_cast<uint32_t(*)[32]>(u));
        tmem_ld32(lane_base + SF_TM_S + grp * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tmem_wait_ld();
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u));
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tc_fence_before();
        mbar_arrive(free_s);
#pragma unroll
        for (int c0 = 0; c0 < 64; ++c0) {
          const float e = ex2(fmaf(__uint_as_float(u[c0]), sl2, nl2));
          pv[c0] = in_range(kbase + c0, lo_i, hi_i) ? e : 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(stP + tile_chunk_off(r, k)) =
            make_uint4(E::pack(pv[8 * k], pv[8 * k + 1]), E::pack(pv[8 * k + 2], pv[8 * k + 3]),
                       E::pack(pv[8 * k + 4], pv[8 * k + 5]), E::pack(pv[8 * k + 6], pv[8 * k + 7]));
      okw = __all_sync(0xffffffffu, mbar_wait(bar_dp, t & 1, abort_flag));
      tc_fence_after();
      {
        uint32_t u[64];
        tmem_ld32(lane_base + SF_TM_DP + grp * 64, *reinterpret_cast<uint32_t(*)[32]>(u));
        tmem_ld32(lane_base + SF_TM_DP + grp * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tmem_wait_ld();
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u));
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tc_fence_before();
        mbar_arrive(free_dp);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c0 = 8 * k + 2 * e;
            // pv is exactly zero outside the mask, so dS is too (for finite dP)
            w[e] = E::pack(pv[c0] * (__uint_as_float(u[c0]) - dl), pv[c0 + 1] * (__uint_as_float(u[c0 + 1]) - dl));
          }
          *reinterpret_cast<uint4*>(stD + tile_chunk_off(r, k)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      if (!named_bar_and(bar_id, 128, okw)) {
        ok = false;
        break;
      }
      if (leader) {
        const long long tix = tile_index(p, b, h, qt, t);
        uint8_t* gp = p.p_tiles + tix * TILE_BYTES + grp * SF_STG;
        uint8_t* gd = p.ds_tiles + tix * TILE_BYTES + grp * SF_STG;
        if (SDPA_ADDR_OK(g.chk, gp, SF_STG)) bulk_store(gp, stP, SF_STG);
        if (SDPA_ADDR_OK(g.chk, gd, SF_STG)) bulk_store(gd, stD, SF_STG);
        bulk_commit_group();
      }
    }
    if (leader) bulk_wait_group0();
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

// ---------------------------------------------------------------------- head_dim 512
// Both passes in one kernel. A 128 x 512 operand is 128 KB, so Q and dO
// cannot both stay in shared memory, nor both in TMEM: Q is copied into TMEM
// (columns 0-255, the A operand of S = Q K^T) and dO stays in shared memory
// (the A operand of dP = dO V^T), which leaves TMEM columns 256-383 for S and
// 384-511 for dP, and 96 KB of shared memory for a ring of six 16 KB K/V
// chunks. Q arrives first in the 128 KB buffer that dO then occupies: the
// epilogue threads copy it into TMEM and only then does the producer load dO
// over it. S and dP are single-buffered but released separately, so S of the
// next key tile is computed while the epilogue waits for dP of this one. Two
// epilogue warpgroups each take 64 keys of a tile and form P and dS in fp32
// (each rounded once); with no shared memory left to stage them, each thread
// stores its row's 16-byte pieces of the two tile images directly. Nothing
// fp32 goes through HBM.
constexpr int S5_CH = 16384;  // ring chunk: 128 rows x 64 columns (one box)
constexpr int S5_NST = 6;
constexpr int S5_A = 8 * S5_CH;  // Q, then dO: eight 64-column atoms
constexpr int S5_NBARS = 2 * S5_NST + 8;
constexpr int S5_SMEM = 1024 + S5_A + S5_NST * S5_CH + S5_NBARS * 8 + 16;
constexpr int S5_THREADS = 320;  // producer, MMA, two epilogue warpgroups (warps 2-5, 6-9)
constexpr int S5_TM_Q = 0, S5_TM_S = 256, S5_TM_DP = 384;
static_assert(S5_SMEM <= 232448, "the head_dim 512 score kernel must fit one CTA's shared memory");

template <bool BF16>
__global__ void __launch_bounds__(S5_THREADS, 1)
    score_fused512_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                          const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ BigBwdParams p) {
  using E = Elem<BF16>;
  const Geom& g = p.g;
  int idx = blockIdx.x + p.item_offset;
  const int h = idx % g.hq;
  idx /= g.hq;
  const int b = idx % g.batch;
  const int qt = p.n_q_tiles - 1 - idx / g.batch;
  const SeqInfo si = seq_info(g, b);
  const int q0 = qt * 128;
  if (q0 >= si.lq) return;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;
  const KeyRange kr = key_range(g, si.lq, si.lk);
  int t_lo, n;
  kv_tiles_of(kr, q0, si.lq, t_lo, n);
  chunk_clip(p, t_lo, n);
  if (n > p.slots) {
    if (threadIdx.x == 0) record_error(p.err, SDPA_ERR_INVALID_ARG);
    return;
  }
  if (n == 0) return;
  const int qhead = si.qhead0 + h;
  const int khead = si.khead0 + h / (g.hq / g.hkv);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;                // Q, then dO
  uint8_t* sRing = sA + S5_A;
  uint64_t* full = reinterpret_cast<uint64_t*>(sRing + S5_NST * S5_CH);
  uint64_t* empty = full + S5_NST;
  uint64_t* bar_qa = empty + S5_NST;  // Q has landed in sA
  uint64_t* bar_q = bar_qa + 1;       // Q is in TMEM (and sA may be overwritten)
  uint64_t* bar_do = bar_q + 1;       // dO has landed in sA
  uint64_t* bar_s = bar_do + 1;       // S of a key tile ready
  uint64_t* bar_dp = bar_s + 1;       // dP of a key tile ready
  uint64_t* free_s = bar_dp + 1;      // the epilogue has read S
  uint64_t* free_dp = free_s + 1;     // ... and dP
  uint64_t* bar_drain = free_dp + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S5_NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(bar_qa, 1);
    mbar_init(bar_q, 256);
    mbar_init(bar_do, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(free_s, 256);
    mbar_init(free_dp, 256);
    mbar_init(bar_drain, 1);
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

  // ring chunk c: key tile c / 16, K columns 64 (c % 16) for c % 16 < 8, then V
  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(bar_qa, S5_A);
      for (int a = 0; a < 8; ++a) tma_load_3d(&tmQ, bar_qa, sA + a * S5_CH, a * 64, qhead, si.qrow0 + q0);
      const int total = 16 * n;
      bool do_issued = false, ok = true;
      int c = 0;
      for (; c < total && ok; ++c) {
        if (c == S5_NST && !do_issued) {
          // the first ring fill is in flight: once Q has left sA, bring dO in
          if (!mbar_wait(bar_q, 0, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_do, S5_A);
          for (int a = 0; a < 8; ++a) tma_load_3d(&tmDO, bar_do, sA + a * S5_CH, a * 64, qhead, si.qrow0 + q0);
          do_issued = true;
        }
        const int slot = c % S5_NST;
        if (!mbar_wait(&empty[slot], ((c / S5_NST) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[slot], S5_CH);
        const int t = c >> 4, kc = c & 15;
        tma_load_3d(kc < 8 ? &tmK : &tmV, &full[slot], sRing + slot * S5_CH, (kc & 7) * 64, khead,
                    si.krow0 + (t_lo + t) * 128);
      }
      if (ok && !do_issued) {  // fewer ring chunks than slots
        if (mbar_wait(bar_q, 0, abort_flag)) {
          mbar_arrive_expect_tx(bar_do, S5_A);
          for (int a = 0; a < 8; ++a) tma_load_3d(&tmDO, bar_do, sA + a * S5_CH, a * 64, qhead, si.qrow0 + q0);
          do_issued = true;
        } else {
          ok = false;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
      const int first = c > S5_NST ? c - S5_NST : 0;
      for (int k = first; k < c; ++k) mbar_wait_drain(&full[k % S5_NST], (k / S5_NST) & 1);
      mbar_wait_drain(bar_qa, 0);
      if (do_issued) mbar_wait_drain(bar_do, 0);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t IDESC = idesc_f16(128, 128, BF16, false, false);
      bool ok = mbar_wait(bar_q, 0, abort_flag);
      tc_fence_after();
      const uint32_t a_base = smem_u32(sA);
      int c = 0;
      for (int t = 0; t < n && ok; ++t) {
        for (int pass = 0; pass < 2 && ok; ++pass) {  // S = Q K^T (A in TMEM), then dP = dO V^T (A in sA)
          if (t >= 1 && !mbar_wait(pass == 0 ? free_s : free_dp, (t - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          if (pass == 1 && t == 0 && !mbar_wait(bar_do, 0, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (pass == 0 ? S5_TM_S : S5_TM_DP);
          for (int kc = 0; kc < 8; ++kc, ++c) {
            const int slot = c % S5_NST;
            if (!mbar_wait(&full[slot], (c / S5_NST) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t bb = smem_u32(sRing + slot * S5_CH);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (pass == 0)
                mma_ts(d, tmem + S5_TM_Q + kc * 32 + ks * 8, smem_desc_sw128(bb + ks * 32, 16, 1024), IDESC,
                       (kc | ks) != 0);
              else
                mma_ss(d, smem_desc_sw128(a_base + kc * S5_CH + ks * 32, 16, 1024),
                       smem_desc_sw128(bb + ks * 32, 16, 1024), IDESC, (kc | ks) != 0);
            }
            mma_commit(&empty[slot]);
          }
          if (ok) mma_commit(pass == 0 ? bar_s : bar_dp);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    }
  } else if (warp >= 2) {
    const int grp = (warp - 2) >> 2;  // 64-key half of each tile; for the TMEM fill, Q atoms 4*grp..
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    const int i = q0 + r;
    const bool valid = i < si.lq;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar_qa, 0, abort_flag));
    if (ok) {
      // row r of Q atoms 4*grp..4*grp+3 -> TMEM columns 32*atom.., packed pairs along D
      for (int a = 4 * grp; a < 4 * grp + 4; ++a) {
        const uint8_t* row = sA + a * S5_CH + r * 128;
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
          v[4 * j] = x.x;
          v[4 * j + 1] = x.y;
          v[4 * j + 2] = x.z;
          v[4 * j + 3] = x.w;
        }
        tmem_st32(lane_base + S5_TM_Q + a * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_q);
    }
    const long long stat = (long long)qhead * p.stat_rows + si.srow0 + i;
    // rows past the sequence end belong to no query: an empty key range, so
    // their P and dS are exactly zero whatever their scores
    const float nl2 = valid && SDPA_ADDR_OK(g.chk, p.nlse2 + stat, 4) ? p.nlse2[stat] : 0.f;
    const float dl = valid && SDPA_ADDR_OK(g.chk, p.delta + stat, 4) ? p.delta[stat] : 0.f;
    const int lo_i = kr.lo(i), hi_i = valid ? kr.hi(i) : lo_i;
    const float sl2 = g.scale_log2;
    for (int t = 0; t < n && ok; ++t) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar_s, t & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kbase = (t_lo + t) * 128 + grp * 64;
      const long long tix = tile_index(p, b, h, qt, t);
      // this thread's row of this group's 64-key atom in the two tile images
      uint8_t* prow = p.p_tiles + tix * TILE_BYTES + grp * 16384 + r * 128;
      uint8_t* drow = p.ds_tiles + tix * TILE_BYTES + grp * 16384 + r * 128;
      const bool prow_ok = SDPA_ADDR_OK(g.chk, prow, 128), drow_ok = SDPA_ADDR_OK(g.chk, drow, 128);
      float pv[64];
      {
        uint32_t u[64];
        tmem_ld32(lane_base + S5_TM_S + grp * 64, *reinterpret_cast<uint32_t(*)[32]>(u));
        tmem_ld32(lane_base + S5_TM_S + grp * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tmem_wait_ld();
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u));
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tc_fence_before();
        mbar_arrive(free_s);
#pragma unroll
        for (int c0 = 0; c0 < 64; ++c0) {
          const float e = ex2(fmaf(__uint_as_float(u[c0]), sl2, nl2));
          pv[c0] = in_range(kbase + c0, lo_i, hi_i) ? e : 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (prow_ok)
          *reinterpret_cast<uint4*>(prow + ((k ^ (r & 7)) << 4)) =
            make_uint4(E::pack(pv[8 * k], pv[8 * k + 1]), E::pack(pv[8 * k + 2], pv[8 * k + 3]),
                       E::pack(pv[8 * k + 4], pv[8 * k + 5]), E::pack(pv[8 * k + 6], pv[8 * k + 7]));
      if (!__all_sync(0xffffffffu, mbar_wait(bar_dp, t & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t u[64];
        tmem_ld32(lane_base + S5_TM_DP + grp * 64, *reinterpret_cast<uint32_t(*)[32]>(u));
        tmem_ld32(lane_base + S5_TM_DP + grp * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tmem_wait_ld();
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u));
        reg_fence(*reinterpret_cast<uint32_t(*)[32]>(u + 32));
        tc_fence_before();
        mbar_arrive(free_dp);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c0 = 8 * k + 2 * e;
            // pv is exactly zero outside the mask, so dS is too (for finite dP)
            w[e] = E::pack(pv[c0] * (__uint_as_float(u[c0]) - dl), pv[c0 + 1] * (__uint_as_float(u[c0 + 1]) - dl));
          }
          if (drow_ok) *reinterpret_cast<uint4*>(drow + ((k ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
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

// ====================================================================== phase 2
// A stage is half a K step: 64 of the 128 contracted rows, i.e. half a tile
// image (16 KB) and 64 rows x 256 columns of B (32 KB). At 48 KB a stage two
// CTAs fit on an SM, so one CTA's prologue and epilogue hide under the other's
// MMAs.
constexpr int GB_STAGE = TILE_BYTES / 2 + 4 * 8192;
constexpr int GB_NST = 2;
constexpr int GB_NBARS = 2 * GB_NST + 3;
constexpr int GB_SMEM = 1024 + GB_NST * GB_STAGE + GB_NBARS * 8 + 16;

// One output tile of one mode. MODE 0: dQ. MODE 1: dV. MODE 2: dK. head: the
// q head (dQ) or kv head (dV/dK); t_own: the tile's own 128-row index (a
// query tile for dQ, a key tile of the chunk for dV/dK); split: its 256-column
// slice of the head dim. tmB is the mode's B operand (K, dO or Q with 64-row
// boxes).
template <int MODE, bool BF16>
__device__ __forceinline__ void gemm_tile(const CUtensorMap* tmB, const BigBwdParams& p, int split, int b, int head,
                                          int t_own) {
  using E = Elem<BF16>;
  using T = typename E::T;
  const Geom& g = p.g;
  const SeqInfo si = seq_info(g, b);
  const int r0 = t_own * 128;
  if (r0 >= (MODE == 0 ? si.lq : si.lk)) return;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;
  const KeyRange kr = key_range(g, si.lq, si.lk);
  const int group = g.hq / g.hkv;
  // K-loop extent
  int t_lo = 0, n = 0, qt_lo = 0, nqt = 0;
  if (MODE == 0) {
    kv_tiles_of(kr, r0, si.lq, t_lo, n);
    chunk_clip(p, t_lo, n);
    // a split key range adds each chunk's part into the accumulator: nothing to add
    if (p.dq_acc && n == 0) return;
  } else {
    const int k_last = min(r0 + 127, si.lk - 1);
    const int qlo = query_lo(kr, r0), qhi = query_hi(kr, k_last, si.lq);
    qt_lo = qlo / 128;
    nqt = qhi > qlo ? (qhi + 127) / 128 - qt_lo : 0;
    n = nqt * group;
  }
  const uint8_t* atiles = MODE == 1 ? p.p_tiles : p.ds_tiles;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + GB_NST * GB_STAGE);
  uint64_t* empty = full + GB_NST;
  uint64_t* bar_done = empty + GB_NST;
  uint64_t* bar_drain = bar_done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // step s of the K-loop: (A tile index, B row start, B generic head)
  auto step = [&](int s, long long& a_tile, int& b_row, int& b_head) {
    if (MODE == 0) {
      a_tile = tile_index(p, b, head, t_own, s);
      b_row = si.krow0 + (t_lo + s) * 128;
      b_head = si.khead0 + head / group;
    } else {
      const int h = head * group + s / nqt;
      const int qt = qt_lo + s % nqt;
      int tl, tn;
      kv_tiles_of(kr, qt * 128, si.lq, tl, tn);
      a_tile = tile_index(p, b, h, qt, t_own - max(tl, p.chunk_lo));
      b_row = si.qrow0 + qt * 128;
      b_head = si.qhead0 + h;
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < GB_NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (elect_one() && n > 0) {
      prefetch_tmap(tmB);
      int s = 0;
      for (; s < 2 * n; ++s) {  // half steps
        const int st = s % GB_NST;
        const int hf = s & 1;
        if (!mbar_wait(&empty[st], ((s / GB_NST) & 1) ^ 1, abort_flag)) break;
        long long at;
        int brow, bh;
        step(s >> 1, at, brow, bh);
        uint8_t* dst = smem + st * GB_STAGE;
        const uint8_t* src = atiles + at * TILE_BYTES;
        mbar_arrive_expect_tx(&full[st], GB_STAGE);
        // a copy the address check rejects still completes its bytes
        auto load = [&](uint8_t* d, const uint8_t* g_src, uint32_t bytes) {
          if (SDPA_ADDR_OK(g.chk, g_src, bytes))
            bulk_load(d, g_src, bytes, &full[st]);
          else
            mbar_complete_tx(&full[st], bytes);
        };
        if (MODE == 0) {  // keys 64*hf.. of the dS image: its atom hf
          load(dst, src + hf * 16384, 16384);
        } else {  // query rows 64*hf.. of the image: the same rows of both atoms
          load(dst, src + hf * 8192, 8192);
          load(dst + 8192, src + 16384 + hf * 8192, 8192);
        }
        for (int a = 0; a < 4; ++a)
          tma_load_3d(tmB, &full[st], dst + TILE_BYTES / 2 + a * 8192, split * 256 + a * 64, bh, brow + hf * 64);
      }
      if (s < 2 * n) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
      for (int k = (s > GB_NST ? s - GB_NST : 0); k < s; ++k) mbar_wait_drain(&full[k % GB_NST], (k / GB_NST) & 1);
    }
  } else if (warp == 1) {
    if (elect_one() && n > 0) {
      // dQ: A = dS tile, K-major (rows = queries). dV/dK: A = P / dS tile read
      // transposed (M = keys, the tile's contiguous dimension). B (K rows for
      // dQ, dO/Q rows for dV/dK) is N-major in every mode.
      constexpr uint32_t IDESC = idesc_f16(128, 256, BF16, MODE != 0, true);
      bool ok = true;
      int s = 0;
      for (; s < 2 * n; ++s) {
        const int st = s % GB_NST;
        if (!mbar_wait(&full[st], (s / GB_NST) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + st * GB_STAGE);
        const uint32_t bb = a + TILE_BYTES / 2;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = MODE == 0 ? smem_desc_sw128(a + ks * 32, 16, 1024)
                                        : smem_desc_sw128(a + ks * 2048, 8192, 1024);
          mma_ss(tmem, ad, smem_desc_sw128(bb + ks * 2048, 8192, 1024), IDESC, (s | ks) != 0);
        }
        mma_commit(&empty[st]);
      }
      if (ok) {
        mma_commit(bar_done);
      } else {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    }
  } else if (warp >= 4) {
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const int row = r0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    bool ok = true;
    if (n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_done, 0, abort_flag));
      tc_fence_after();
    }
    if (!ok) {
      *abort_flag = 1;
      record_error(p.err, SDPA_ERR_TIMEOUT);
    } else {
      T* out;
      float mul;
      bool valid;
      if (MODE == 0) {
        out = reinterpret_cast<T*>(p.dq) + ((long long)(si.qrow0 + row) * g.nh_q + si.qhead0 + head) * g.d;
        mul = g.scale;
        valid = row < si.lq;
      } else {
        out = reinterpret_cast<T*>(MODE == 1 ? p.dv : p.dk) +
              ((long long)(si.krow0 + row) * g.nh_kv + si.khead0 + head) * g.d;
        mul = MODE == 2 ? g.scale : 1.f;
        valid = row < si.lk;
      }
      out += split * 256;
      if (MODE == 0 && p.dq_acc) {
        // key range split into chunks: add this chunk's unscaled part into the
        // head-major fp32 accumulator (the dQ finalise scales and converts it)
        float* acc = p.dq_acc + ((long long)(si.qhead0 + head) * g.rows_q + si.qrow0 + row) * g.d + split * 256;
#pragma unroll 1
        for (int c = 0; c < 256 / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(lane_base + c * 32, u);
          tmem_wait_ld();
          reg_fence(u);
          if (valid && SDPA_ADDR_OK(g.chk, acc + c * 32, 128)) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              red_add_v4_f32(acc + c * 32 + 4 * e, __uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                             __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]));
          }
        }
      } else {
#pragma unroll 1
      for (int c = 0; c < 256 / 32; ++c) {
        uint32_t packed[16];
        if (n > 0) {
          uint32_t u[32];
          tmem_ld32(lane_base + c * 32, u);
          tmem_wait_ld();
          reg_fence(u);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            packed[e] = E::pack(__uint_as_float(u[2 * e]) * mul, __uint_as_float(u[2 * e + 1]) * mul);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) packed[e] = 0u;
        }
        if (valid && SDPA_ADDR_OK(g.chk, out + c * 32, 64)) {
          uint4* d4 = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
        }
      }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Phase 2 of one chunk in one launch. The three modes only read the chunk's
// P / dS images and Q, dO, K, so they run side by side. Two grid orders:
//  * by mode (unbounded masks): dV and dK of every key tile of the chunk, then
//    dQ of every query tile. A dK/dV CTA loops over every query tile of its
//    group, several times a dQ CTA's key tiles, and these long CTAs start first.
//  * by (batch, kv head) block (a bounded window): a block holds dV and dK of
//    the chunk's key tiles, then dQ of its query tiles for the q heads of the
//    group. The window keeps a block's dS band small, so dQ reads the images
//    dK has just read while they are still in L2; the CTAs are of similar
//    length.
template <bool BF16>
__global__ void __launch_bounds__(256, 2)
    gemm_kernel(const __grid_constant__ CUtensorMap tmK64, const __grid_constant__ CUtensorMap tmDO64,
                const __grid_constant__ CUtensorMap tmQ64, const __grid_constant__ BigBwdParams p, int n_q_tiles) {
  const Geom& g = p.g;
  const int splits = g.d / 256, group = g.hq / g.hkv;
  const int n_kv = p.chunk_hi - p.chunk_lo;
  int idx = blockIdx.x + p.item_offset;
  if (p.block_major) {
    const int kv_ctas = 2 * splits * n_kv;
    const int per_block = kv_ctas + group * splits * n_q_tiles;
    int r = idx % per_block;
    idx /= per_block;
    const int kvh = idx % g.hkv;
    const int b = idx / g.hkv;
    if (r < kv_ctas) {  // dV and dK of key tile chunk_lo + r / (2 * splits)
      const int t = r / (2 * splits);
      r %= 2 * splits;
      if (r < splits)
        gemm_tile<1, BF16>(&tmDO64, p, r, b, kvh, p.chunk_lo + t);
      else
        gemm_tile<2, BF16>(&tmQ64, p, r - splits, b, kvh, p.chunk_lo + t);
    } else {  // dQ of query tile t for the q heads of the group
      r -= kv_ctas;
      const int t = r / (group * splits);
      r %= group * splits;
      gemm_tile<0, BF16>(&tmK64, p, r % splits, b, kvh * group + r / splits, t);
    }
    return;
  }
  // by mode: every dV tile (key tile fastest), every dK tile, then every dQ
  // tile (heaviest query tiles first)
  const int kv_mode = n_kv * splits * g.hkv * g.batch;
  if (idx < 2 * kv_mode) {
    const bool dk = idx >= kv_mode;
    int x = dk ? idx - kv_mode : idx;
    const int t = x % n_kv;
    x /= n_kv;
    const int split = x % splits;
    x /= splits;
    if (dk)
      gemm_tile<2, BF16>(&tmQ64, p, split, x / g.hkv, x % g.hkv, p.chunk_lo + t);
    else
      gemm_tile<1, BF16>(&tmDO64, p, split, x / g.hkv, x % g.hkv, p.chunk_lo + t);
  } else {
    int x = idx - 2 * kv_mode;
    const int split = x % splits;
    x /= splits;
    const int head = x % g.hq;
    x /= g.hq;
    const int b = x % g.batch;
    gemm_tile<0, BF16>(&tmK64, p, split, b, head, n_q_tiles - 1 - x / g.batch);
  }
}

// ====================================================================== launch
template <class K>
static bool set_smem(K kern, int bytes) {
  return set_kernel_smem(reinterpret_cast<const void*>(kern), bytes, 100) == SDPA_OK;
}

template <int DQK, bool BF16>
static int launch_big_t(const BigBwdLaunch& L, int* launches) {
  const BigBwdParams& p0 = L.p;
  const int splits = p0.g.d / 256;
  const long long g1 = (long long)p0.n_q_tiles * p0.g.hq * p0.g.batch;
  const long long gq = g1 * splits;
  const long long gkv = (long long)std::min(p0.chunk, p0.n_kv_tiles) * splits * p0.g.hkv * p0.g.batch;
  if (g1 > 0x7fffffffLL || gq + 2 * gkv > 0x7fffffffLL) return SDPA_ERR_UNSUPPORTED;
  if (p0.chunk <= 0 || (p0.chunk < p0.n_kv_tiles && !p0.dq_acc)) return SDPA_ERR_INVALID_ARG;
  auto gm = gemm_kernel<BF16>;
  if (!set_smem(gm, GB_SMEM)) return SDPA_ERR_CUDA;
  auto sf = DQK == 256 ? score_fused256_kernel<BF16> : score_fused512_kernel<BF16>;
  const int sf_smem = DQK == 256 ? SF_SMEM : S5_SMEM;
  const int sf_threads = DQK == 256 ? SF_THREADS : S5_THREADS;
  if (!set_smem(sf, sf_smem)) return SDPA_ERR_CUDA;
  int n = 0;
  // one chunk of key tiles at a time: phase 1 writes its P / dS tiles, phase 2
  // consumes them before the next chunk's phase 1 overwrites the arrays
  for (int lo = 0; lo < p0.n_kv_tiles; lo += p0.chunk) {
    BigBwdParams p = p0;
    p.chunk_lo = lo;
    p.chunk_hi = std::min(lo + p0.chunk, p0.n_kv_tiles);
    int rc = SDPA_OK;
    if (g1 > 0) {  // phase 1: P and dS tiles of this chunk from S and dP
      rc = launch_in_grids(g1, [&](long long off, long long cnt) {
        BigBwdParams pp = p;
        pp.item_offset = (int)off;
        sf<<<(unsigned)cnt, sf_threads, sf_smem, L.stream>>>(L.tmQ, L.tmDO, L.tmK, L.tmV, pp);
        ++n;
        return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
      });
      if (rc) return rc;
    }
    const int nq2 = g1 > 0 ? p.n_q_tiles : 0;  // query tiles whose dQ part this chunk adds
    p.block_major = p.g.wl >= 0;
    const long long g2 = ((long long)2 * (p.chunk_hi - p.chunk_lo) + (long long)(p.g.hq / p.g.hkv) * nq2) * splits *
                         p.g.hkv * p.g.batch;
    if (g2 > 0x7fffffffLL) return SDPA_ERR_UNSUPPORTED;
    if (g2 > 0) {  // phase 2: dV, dK of the chunk's key tiles, its part of dQ
      rc = launch_in_grids(g2, [&](long long off, long long cnt) {
        BigBwdParams pp = p;
        pp.item_offset = (int)off;
        gm<<<(unsigned)cnt, 256, GB_SMEM, L.stream>>>(L.tmK64, L.tmDO64, L.tmQ64, pp, nq2);
        ++n;
        return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
      });
      if (rc) return rc;
    }
  }
  *launches = n;
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

int launch_bwd_big(const BigBwdLaunch& L, int head_dim, bool bf16, int* launches) {
  *launches = 0;
  if (head_dim == 256) return bf16 ? launch_big_t<256, true>(L, launches) : launch_big_t<256, false>(L, launches);
  if (head_dim == 512) return bf16 ? launch_big_t<512, true>(L, launches) : launch_big_t<512, false>(L, launches);
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace sdpa
