// bwd.cu -- fused attention backward for sm_103a, head_dim 128.
//
// One CTA owns one 128-key tile of one (batch, kv head). K and V stay in
// shared memory; the CTA walks every q head of the GQA group and every
// 64-row query tile that can attend its keys, so dK and dV accumulate in
// TMEM without atomics. Per query tile (all MMAs tcgen05, fp32 in TMEM):
//   S^T  = K Q^T                 (SS, M=128 keys, N=64 queries)
//   dP^T = V dO^T                (SS)
//   softmax warps: P^T = exp2(S^T*scale*log2e - LSE*log2e), masked,
//                  dS^T = P^T * (dP^T - delta); both written back to TMEM as
//                  16-bit values, dS^T also to shared memory
//   dV  += P^T dO                (TS, A = P^T from TMEM)
//   dK  += dS^T Q                (TS)
//   dQ^T = K^T dS^T              (SS, M=128 head-dim rows, N=64 queries)
//   drain warps: dQ^T -> shared memory -> bulk reduce-add (fp32) into the
//                head-major dQ accumulator; a finalise kernel scales and casts.
// S^T and dP^T are double-buffered in TMEM: while the softmax warps work on
// step i, the tensor pipe runs dV/dK/dQ of step i-1 and S^T/dP^T of step i+1,
// so the softmax is the only serial link. dQ^T of step i lands in step i's
// dP^T/dS^T columns (dK has consumed dS^T by then), so S^T of step i+2 can
// follow at once; only dP^T of step i+2 waits for the drain to read dQ^T. dQ accumulation uses no inter-CTA
// barriers or credits: every contribution is an independent fp32 reduction.
//
// Roles (512 threads): warp 0 TMA producer; warp 1 TMEM allocator + MMA
// issuer; warps 4-7 and 8-11 softmax (one thread per key row, each
// warpgroup one half of the 64 query columns) and the dV / dK epilogue;
// warps 12-15 dQ drain (one thread per head-dim row).
// TMEM: dV [0,128) dK [128,256) S^T/P^T [256,320) [320,384)
//       dP^T/dS^T(/dQ^T) [384,448) [448,512).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr int BN = 128;  // keys per CTA
constexpr int BQ = 64;   // queries per step
constexpr int D = 128;
constexpr int K_BYTES = BN * D * 2;   // 32 KB, two 64-column atoms of 16 KB
constexpr int QT_BYTES = BQ * D * 2;  // 16 KB, two atoms of 8 KB
constexpr int STAT_FLOATS = BQ;       // a query tile's rows: one aligned block (SeqInfo::srow0)
constexpr int NQS = 3;                // Q/dO stages
constexpr int DS_BYTES = BN * BQ * 2; // 16 KB
constexpr int STG_BYTES = BQ * D * 4; // 32 KB fp32 dQ staging

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + K_BYTES;
constexpr int OFF_Q = OFF_V + K_BYTES;                   // NQS x 16 KB
constexpr int OFF_DO = OFF_Q + NQS * QT_BYTES;           // NQS x 16 KB
constexpr int OFF_DS = OFF_DO + NQS * QT_BYTES;          // 2 x 16 KB
constexpr int OFF_STG = OFF_DS + 2 * DS_BYTES;           // 32 KB
constexpr int OFF_STAT = OFF_STG + STG_BYTES;            // NQS x (lse2, delta) x 68 floats
constexpr int OFF_BAR = OFF_STAT + NQS * 2 * STAT_FLOATS * 4;
constexpr int NBARS = 2 * NQS + 10;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBARS * 8 + 16;

// S^T/P^T and dP^T/dS^T are double-buffered; dQ^T of step i is written into
// step i's dP^T/dS^T columns once dK(i) has consumed dS^T.
constexpr uint32_t TM_DV = 0, TM_DK = 128;
__device__ __forceinline__ uint32_t tm_s(int buf) { return 256u + 64u * buf; }
__device__ __forceinline__ uint32_t tm_dp(int buf) { return 384u + 64u * buf; }

// Column (within a 64-column S^T/dP^T buffer) of the packed 16-bit operand
// for queries [16*ks, 16*ks+16): each half of 32 queries is packed into the
// first 16 columns of its own 32.
__device__ __forceinline__ uint32_t p_col(int ks) { return (uint32_t)((ks >> 1) * 32 + (ks & 1) * 8); }

// P^T and dS^T for 32 query columns of one key row:
//   P = exp2(S * scale*log2e - LSE*log2e) (zero where masked),
//   dS = P * (dP - delta), both packed to 16-bit pairs.
// nl2 holds -LSE*log2e (-inf for rows without keys), dl the deltas; both are
// 16-byte aligned in shared memory and read four at a time (the same address
// for the whole warp, so one 16-byte broadcast feeds four columns).
template <bool MASK, class E>
__device__ __forceinline__ void p_ds_cols(const uint32_t (&us)[32], const uint32_t (&ud)[32], const float* nl2,
                                          const float* dl, float sl2, int q, int qlo, int qhi, uint32_t (&pp)[16],
                                          uint32_t (&pd)[16]) {
  const float2 sc = make_float2(sl2, sl2);
#pragma unroll
  for (int c4 = 0; c4 < 32; c4 += 4) {
    const float4 n4 = *reinterpret_cast<const float4*>(nl2 + c4);
    const float4 d4 = *reinterpret_cast<const float4*>(dl + c4);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c4 + 2 * h;
      const float2 nn = h ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y);
      const float2 dd = h ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
      const float2 t = ffma2(make_float2(__uint_as_float(us[c]), __uint_as_float(us[c + 1])), sc, nn);
      float p0 = ex2(t.x), p1 = ex2(t.y);
      if (MASK) {
        p0 = in_range(q + c, qlo, qhi) ? p0 : 0.f;
        p1 = in_range(q + c + 1, qlo, qhi) ? p1 : 0.f;
      }
      const float2 d = fsub2(make_float2(__uint_as_float(ud[c]), __uint_as_float(ud[c + 1])), dd);
      const float2 ds = fmul2(make_float2(p0, p1), d);
      pp[c / 2] = E::pack(p0, p1);
      pd[c / 2] = E::pack(ds.x, ds.y);
    }
  }
}

}  // namespace

// DQ = false: dK and dV only (no dS^T copy, no dQ^T MMA, no drain).
template <bool BF16, bool DQ>
__global__ void __launch_bounds__(512, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ BwdParams p) {
  using E = Elem<BF16>;
  using T = typename E::T;
  const Geom& g = p.g;

  // ---- which tile. Grid order: sequence (THD: longest first, through the
  // order the guard kernel wrote), then blocks of head_block kv heads, then
  // key tile, then kv head within the block. A key tile is attended by no
  // more query tiles than the tile before it under every supported mask, so
  // each sequence's heaviest CTAs start first and the grid ends on light
  // ones; the key tiles of one (sequence, kv head) start close together and
  // walk the same Q/dO rows and dQ accumulator rows while those are resident
  // in L2 (head_block bounds how many heads' rows are in use at once).
  int idx = blockIdx.x + p.item_offset;
  const int per_seq = p.n_kv_tiles * g.hkv;
  const int hb = p.head_block;
  int b = idx / per_seq;
  idx %= per_seq;
  const int blk = idx / (p.n_kv_tiles * hb);
  idx %= p.n_kv_tiles * hb;
  const int kt = idx / hb;
  const int kvh = blk * hb + idx % hb;
  if (p.order) b = SDPA_ADDR_OK(g.chk, p.order + b, 4) ? p.order[b] : -1;
  if (kvh >= g.hkv || (unsigned)b >= (unsigned)g.batch) {
    if (threadIdx.x == 0) record_error(p.err, SDPA_ERR_INVALID_ARG);
    return;
  }
  const SeqInfo si = seq_info(g, b);
  const int k0 = kt * BN;
  if (k0 >= si.lk) return;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;

  const KeyRange kr = key_range(g, si.lq, si.lk);
  const int k_last = min(k0 + BN - 1, si.lk - 1);
  const int qlo = query_lo(kr, k0), qhi = query_hi(kr, k_last, si.lq);
  const int qt_lo = qlo / BQ;
  const int nqt = qhi > qlo ? (qhi + BQ - 1) / BQ - qt_lo : 0;
  const int group = g.hq / g.hkv;
  const int n = nqt * group;
  const int khead = si.khead0 + kvh;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
  float* sstat = reinterpret_cast<float*>(smem + OFF_STAT);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;            // [NQS]
  uint64_t* empty = bars + NQS;     // [NQS]
  uint64_t* bar_kv = bars + 2 * NQS;
  uint64_t* bar_sdp = bar_kv + 1;     // [2] S^T, dP^T of a step ready (per buffer)
  uint64_t* bar_ds = bar_sdp + 2;     // softmax of a step done
  uint64_t* bar_dq = bar_ds + 1;      // [2] dQ^T of a step ready (per buffer)
  uint64_t* bar_dqfree = bar_dq + 2;  // drain has read dQ^T of a step
  uint64_t* bar_final = bar_dqfree + 1;
  uint64_t* bar_drain = bar_final + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // (head in group, query tile) of step i
  auto step_head = [&](int i) { return kvh * group + i / nqt; };
  auto step_q0 = [&](int i) { return (qt_lo + i % nqt) * BQ; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NQS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(bar_kv, 1);
    mbar_init(&bar_sdp[0], 1);
    mbar_init(&bar_sdp[1], 1);
    mbar_init(bar_ds, 256);
    mbar_init(&bar_dq[0], 1);
    mbar_init(&bar_dq[1], 1);
    mbar_init(bar_dqfree, 128);
    mbar_init(bar_final, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one() && n > 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmDO);
      mbar_arrive_expect_tx(bar_kv, 2 * K_BYTES);
      const int krow = si.krow0 + k0;
      tma_load_3d(&tmK, bar_kv, smem + OFF_K, 0, khead, krow);
      tma_load_3d(&tmK, bar_kv, smem + OFF_K + 16384, 64, khead, krow);
      tma_load_3d(&tmV, bar_kv, smem + OFF_V, 0, khead, krow);
      tma_load_3d(&tmV, bar_kv, smem + OFF_V + 16384, 64, khead, krow);
      int i = 0;
      for (; i < n; ++i) {
        const int st = i % NQS;
        if (!mbar_wait(&empty[st], ((i / NQS) & 1) ^ 1, abort_flag)) break;
        const int qhead = si.qhead0 + step_head(i);
        const int row0 = si.qrow0 + step_q0(i);
        mbar_arrive_expect_tx(&full[st], 2 * QT_BYTES + 2 * STAT_FLOATS * 4);
        uint8_t* sq = smem + OFF_Q + st * QT_BYTES;
        uint8_t* sd = smem + OFF_DO + st * QT_BYTES;
        tma_load_3d(&tmQ, &full[st], sq, 0, qhead, row0);
        tma_load_3d(&tmQ, &full[st], sq + 8192, 64, qhead, row0);
        tma_load_3d(&tmDO, &full[st], sd, 0, qhead, row0);
        tma_load_3d(&tmDO, &full[st], sd + 8192, 64, qhead, row0);
        const long long so = (long long)qhead * p.stat_rows + si.srow0 + step_q0(i);
        if (SDPA_ADDR_OK(g.chk, p.lse2 + so, STAT_FLOATS * 4))
          bulk_load(sstat + st * 2 * STAT_FLOATS, p.lse2 + so, STAT_FLOATS * 4, &full[st]);
        else
          mbar_complete_tx(&full[st], STAT_FLOATS * 4);
        if (SDPA_ADDR_OK(g.chk, p.delta + so, STAT_FLOATS * 4))
          bulk_load(sstat + st * 2 * STAT_FLOATS + STAT_FLOATS, p.delta + so, STAT_FLOATS * 4, &full[st]);
        else
          mbar_complete_tx(&full[st], STAT_FLOATS * 4);
      }
      if (i < n) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
      mbar_wait_drain(bar_kv, 0);
      for (int k = (i > NQS ? i - NQS : 0); k < i; ++k) mbar_wait_drain(&full[k % NQS], (k / NQS) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one() && n > 0) {
      constexpr uint32_t ID_S = idesc_f16(128, BQ, BF16, false, false);     // S^T, dP^T
      constexpr uint32_t ID_KV = idesc_f16(128, D, BF16, false, true);      // dV, dK (B = dO/Q, N-major)
      constexpr uint32_t ID_DQ = idesc_f16(128, BQ, BF16, true, true);      // dQ^T (A = K^T, B = dS^T)
      const uint32_t sK = smem_u32(smem + OFF_K), sV = smem_u32(smem + OFF_V);
      bool ok = mbar_wait(bar_kv, 0, abort_flag);
      // S^T(i) = K Q^T into its buffer (after the Q/dO stage of step i landed)
      auto issue_s = [&](int i) -> bool {
        const int st = i % NQS;
        if (!mbar_wait(&full[st], (i / NQS) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t sq = smem_u32(smem + OFF_Q + st * QT_BYTES);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ka = (ks >> 2) * 16384 + (ks & 3) * 32;
          const uint32_t qa = (ks >> 2) * 8192 + (ks & 3) * 32;
          mma_ss(tmem + tm_s(i & 1), smem_desc_sw128(sK + ka, 16, 1024), smem_desc_sw128(sq + qa, 16, 1024), ID_S,
                 ks > 0);
        }
        return true;
      };
      // dP^T(i) = V dO^T (the stage is known to have landed), then signal S^T/dP^T(i)
      auto issue_dp = [&](int i) {
        const int st = i % NQS;
        const uint32_t sd = smem_u32(smem + OFF_DO + st * QT_BYTES);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ka = (ks >> 2) * 16384 + (ks & 3) * 32;
          const uint32_t qa = (ks >> 2) * 8192 + (ks & 3) * 32;
          mma_ss(tmem + tm_dp(i & 1), smem_desc_sw128(sV + ka, 16, 1024), smem_desc_sw128(sd + qa, 16, 1024), ID_S,
                 ks > 0);
        }
        mma_commit(&bar_sdp[i & 1]);
      };
      auto wait_ds = [&](int i) -> bool {
        if (!mbar_wait(bar_ds, i & 1, abort_flag)) return false;
        tc_fence_after();
        return true;
      };
      // dV += P^T(i) dO(i)
      auto issue_dv = [&](int i) {
        const uint32_t sd = smem_u32(smem + OFF_DO + (i % NQS) * QT_BYTES);
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks)
          mma_ts(tmem + TM_DV, tmem + tm_s(i & 1) + p_col(ks), smem_desc_sw128(sd + ks * 2048, 8192, 1024), ID_KV,
                 (i | ks) != 0);
      };
      // dK += dS^T(i) Q(i); the Q/dO stage of step i is then free
      auto issue_dk = [&](int i) {
        const int st = i % NQS;
        const uint32_t sq = smem_u32(smem + OFF_Q + st * QT_BYTES);
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks)
          mma_ts(tmem + TM_DK, tmem + tm_dp(i & 1) + p_col(ks), smem_desc_sw128(sq + ks * 2048, 8192, 1024), ID_KV,
                 (i | ks) != 0);
        mma_commit(&empty[st]);
      };
      // dQ^T(i) into the dP^T/dS^T columns dK(i) has just read
      auto issue_dq = [&](int i) {
        const uint32_t sds = smem_u32(smem + OFF_DS + (i & 1) * DS_BYTES);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_ss(tmem + tm_dp(i & 1), smem_desc_sw128(sK + ks * 2048, 16384, 1024),
                 smem_desc_sw128(sds + ks * 2048, 16384, 1024), ID_DQ, ks > 0);
        mma_commit(&bar_dq[i & 1]);
      };
      // Issue stream: ... dQ^T(i), S^T(i+2), dV(i+1), [drain has read dQ^T(i)] dP^T(i+2), dK(i+1),
      // dQ^T(i+1), S^T(i+3), dV(i+2), ... Each write follows every read of the
      // columns it overwrites in issue order (S^T(i+2) after dV(i), dP^T(i+2)
      // after dK(i) and the drain of dQ^T(i), dQ^T(i+1) after dK(i+1)), the
      // drain of dQ^T(i) is covered by S^T(i+2) and dV(i+1), and the softmax of
      // step i+2 by dK(i+1), dQ^T(i+1) and S^T(i+3).
      tc_fence_after();
      for (int i = 0; i < 2 && i < n && ok; ++i) {
        ok = issue_s(i);
        if (ok) issue_dp(i);
      }
      if (ok && n > 0) {
        ok = wait_ds(0);
        if (ok) {
          issue_dv(0);
          issue_dk(0);
          if (DQ) issue_dq(0);
          if (n > 2) ok = issue_s(2);
        }
      }
      for (int i = 0; i < n && ok; ++i) {
        if (i + 1 < n) {
          if (!(ok = wait_ds(i + 1))) break;
          issue_dv(i + 1);
        }
        if (i + 2 < n) {
          if (DQ && !mbar_wait(bar_dqfree, i & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_dp(i + 2);
        }
        if (i + 1 < n) {
          issue_dk(i + 1);
          if (DQ) issue_dq(i + 1);
          if (i + 3 < n && !(ok = issue_s(i + 3))) break;
        }
      }
      if (ok) {
        mma_commit(bar_final);
      } else {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax
    // Two warpgroups split the 64 query columns of a step: warpgroup `half`
    // owns columns [32*half, 32*half+32). Each writes its packed P^T / dS^T
    // into the first 16 of its own 32 columns, so neither overwrites scores
    // the other has not read yet.
    const int half = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row in the tile
    const int j = k0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = g.scale_log2;
    const bool key_ok = j < si.lk;
    const int my_qlo = key_ok ? query_lo(kr, j) : 0;
    const int my_qhi = key_ok ? query_hi(kr, j, si.lq) : 0;
    const int lo_last = query_lo(kr, k_last), hi_first = query_hi(kr, k0, si.lq);
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int st = i % NQS;
      const int q0 = step_q0(i);
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_sdp[buf], (i >> 1) & 1, abort_flag) &&
                                       mbar_wait(&full[st], (i / NQS) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool interior = (k0 + BN <= si.lk) && (q0 + BQ <= si.lq) && lo_last <= q0 && hi_first >= q0 + BQ;
      const float* nl2 = sstat + st * 2 * STAT_FLOATS + half * 32;
      const float* dl = nl2 + STAT_FLOATS;
      uint32_t us[32], ud[32];
      tmem_ld32(lane_base + tm_s(buf) + half * 32, us);
      tmem_ld32(lane_base + tm_dp(buf) + half * 32, ud);
      tmem_wait_ld();
      reg_fence(us);
      reg_fence(ud);
      uint32_t pp[16], pd[16];
      if (interior)
        p_ds_cols<false, E>(us, ud, nl2, dl, sl2, 0, 0, 0, pp, pd);
      else
        p_ds_cols<true, E>(us, ud, nl2, dl, sl2, q0 + half * 32, my_qlo, my_qhi, pp, pd);
      tmem_st16(lane_base + tm_s(buf) + half * 32, pp);
      tmem_st16(lane_base + tm_dp(buf) + half * 32, pd);
      if (DQ) {
        // dS^T row r, queries [32*half, 32*half+32): four 16-byte chunks placed
        // with the 128-byte swizzle (chunk ^ (row % 8)).
        uint8_t* ds_row = smem + OFF_DS + buf * DS_BYTES + r * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = half * 4 + k;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) * 16)) =
              make_uint4(pd[4 * k], pd[4 * k + 1], pd[4 * k + 2], pd[4 * k + 3]);
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ds);
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_final, 0, abort_flag));
      tc_fence_after();
    }
    if (!ok) {
      *abort_flag = 1;
      record_error(p.err, SDPA_ERR_TIMEOUT);
    } else {
      // warpgroup 0 stores dV, warpgroup 1 stores dK (scaled)
      T* dst = reinterpret_cast<T*>(half ? p.dk : p.dv) + ((long long)(si.krow0 + j) * g.nh_kv + khead) * D;
      const float mul = half ? g.scale : 1.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t packed[16];
        if (n > 0) {
          uint32_t u[32];
          tmem_ld32(lane_base + (half ? TM_DK : TM_DV) + c * 32, u);
          tmem_wait_ld();
          reg_fence(u);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            packed[e] = E::pack(__uint_as_float(u[2 * e]) * mul, __uint_as_float(u[2 * e + 1]) * mul);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) packed[e] = 0u;
        }
        if (key_ok && SDPA_ADDR_OK(g.chk, dst + c * 32, 64)) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
        }
      }
    }
  } else if (warp >= 12 && DQ) {
    // ------------------------------------------------------------ dQ drain
    const int wq = warp & 3;
    const int dcol = wq * 32 + lane;  // head-dim row of dQ^T
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    float* stg = reinterpret_cast<float*>(smem + OFF_STG);
    const bool leader = threadIdx.x == 384;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_dq[buf], (i >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t u0[32], u1[32];
      tmem_ld32(lane_base + tm_dp(buf), u0);
      tmem_ld32(lane_base + tm_dp(buf) + 32, u1);
      tmem_wait_ld();
      reg_fence(u0);
      reg_fence(u1);
      tc_fence_before();
      mbar_arrive(bar_dqfree);
      if (leader) bulk_wait_group_read0();
      named_bar_sync(1, 128);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        stg[c * D + dcol] = __uint_as_float(u0[c]);
        stg[(32 + c) * D + dcol] = __uint_as_float(u1[c]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (leader) {
        const int q0 = step_q0(i);
        const int rows = min(BQ, si.lq - q0);
        if (rows > 0) {
          const int qhead = si.qhead0 + step_head(i);
          float* dstp = p.dq_acc + ((long long)qhead * g.rows_q + si.qrow0 + q0) * D;
          if (SDPA_ADDR_OK(g.chk, dstp, rows * D * 4)) bulk_reduce_add_f32(dstp, stg, rows * D * 4);
          bulk_commit_group();
        }
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

template <bool BF16, bool DQ>
static int launch_t(const BwdLaunch& L) {
  auto kern = bwd_kernel<BF16, DQ>;
  if (const int rc = set_kernel_smem(reinterpret_cast<const void*>(kern), SMEM_BYTES, -1)) return rc;
  const long long grid = (long long)L.p.n_kv_tiles * L.p.g.hkv * L.p.g.batch;
  if (grid <= 0) return SDPA_OK;
  if (grid > 0x7fffffffLL) return SDPA_ERR_UNSUPPORTED;
  return launch_in_grids(grid, [&](long long off, long long n) {
    BwdParams p = L.p;
    p.item_offset = (int)off;
    kern<<<(unsigned)n, 512, SMEM_BYTES, L.stream>>>(L.tmQ, L.tmK, L.tmV, L.tmDO, p);
    return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
  });
}

int launch_bwd_dkdv(const BwdLaunch& L, int head_dim, bool bf16, bool with_dq, int* launches) {
  *launches = 0;
  if (head_dim != 128) return SDPA_ERR_UNSUPPORTED;
  const int rc = with_dq ? (bf16 ? launch_t<true, true>(L) : launch_t<false, true>(L))
                         : (bf16 ? launch_t<true, false>(L) : launch_t<false, false>(L));
  if (rc == SDPA_OK) *launches = 1;
  return rc;
}

}  // namespace sdpa
