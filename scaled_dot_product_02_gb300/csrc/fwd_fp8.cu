// fwd_fp8.cu -- FP8 (E4M3) attention forward for sm_103a, head_dim 128 and 256.
//
// Reading of TransformerEngine PR #3705's closing note on FP8 ("Amax S"):
// with E4M3 inputs the softmax output is stored in E4M3 under the fixed
// scale 448 (the format's largest value; no dropout), so no amax of it is
// needed -- which holds when the stored probabilities are normalised by the
// row's largest. Q, K, V are E4M3 codes with per-tensor descales d_q, d_k, d_v:
//   S   = scale * d_q * d_k * Q8 K8^T            (tcgen05 kind::f8f6f4, fp32)
//   m   = max_j S_ij (masked),  P~ = exp(S - m) <= 1,  l = sum_j P~_ij
//   P8  = E4M3(P~ * 448)                          (round to nearest even)
//   O   = P8 V8 * d_v / (448 * l),  LSE = m + ln l
// The kernel makes two passes over the keys of a query tile: pass 1 computes
// S for every key tile and keeps only the row max (no exponentials); pass 2
// computes S again, forms P~ against the final max, sums it, rounds it to
// E4M3 into TMEM and accumulates P8 V there. The extra S costs 2*D flop per
// pair at the 8-bit rate; in exchange P is rounded on the definition's own
// grid, exp runs once per score, and O is never rescaled.
//
// Operands are K-major 128-byte-swizzled E4M3 tiles (128 rows x 128 bytes,
// 16 KB): Q and K straight from their [row][head][128] tensors, and V from a
// transposed copy Vt[head][d][key] that vt_kernel writes into the workspace
// on every call (V is key-major in memory; as the B operand of P V it must
// be contracted over keys). Each sequence's keys start on a 16-byte boundary
// of Vt (TMA's alignment rule for the innermost coordinate), and the gaps
// between sequences hold zeros.
//
// The kernel is persistent (one CTA per SM), tiles taken heaviest first from
// an atomic ticket counter. At head_dim 128 it runs two query-tile pipelines.
// Roles (384 threads): warps 0-3 / 4-7 softmax and epilogue of pipeline 0 / 1
// (one thread per query row, all 128 keys of a step), warps 8 / 9 TMA
// producer and scheduler of pipeline 0 / 1, warp 10 TMEM allocator and MMA
// issuer serving the two pipelines strictly in turn (so one pipeline's
// softmax runs under the other's MMAs), warp 11 completes the third
// warpgroup. Per pipeline: a Q tile and a four-stage K / Vt ring in shared
// memory; in TMEM its O (128 columns) and one S buffer (128), into whose
// first 32 columns the softmax writes P8 for the P8 V MMA.
// At head_dim 256 O takes 256 TMEM columns, so there is one pipeline with two
// S buffers: step u of a tile runs in buffer u % 2 on softmax warpgroup
// u % 2, and S of step u + 2 is computed while the other warpgroup works on
// step u + 1. Pass 2 needs no running max (the max is final), so the two
// warpgroups' steps are independent; they exchange their partial row maxima
// before pass 2 and their row sums before the epilogue (shared memory, an
// mbarrier each), and each stores half of O.
// On unmasked key tiles pass 1 takes each 32-column chunk's max from the TMEM
// load itself (load with max reduction).
#include <algorithm>

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr int F8_BM = 128, F8_BN = 128;
// Per head_dim D (128 or 256): two query-tile pipelines at D = 128 (as the
// head_dim 128 bf16 forward), one at D = 256 (its O takes 256 TMEM columns).
// Each pipeline has its Q tile, a ring of NST K / Vt tiles and, in TMEM, its
// O (D columns) and one S buffer (128; P8 is written back into it for the
// P8 V MMA). A Q or K tile is D / 128 atoms of 128 rows x 128 one-byte
// columns; a Vt tile is D rows of 128 keys.
template <int D>
struct F8Cfg {
  static constexpr int NPIPE = D == 128 ? 2 : 1;
  // softmax warpgroups per pipeline: at D = 256 both serve the one pipeline,
  // taking its steps in turn, each with its own S buffer
  static constexpr int NSM = D == 128 ? 1 : 2;
  static constexpr int ATOMS = D / 128;
  static constexpr int TILE = 128 * D;  // bytes of a Q, K or Vt tile
  static constexpr int NST = 4;
  static constexpr int PIPE_BYTES = TILE + NST * TILE;  // per pipeline, 1024-aligned
  static constexpr int PIPE_BARS = 2 * NST + 16;         // mbarriers + queue per pipeline (8 bytes each)
  static constexpr int STG_BYTES = 8 * 2048;  // per softmax warp: 32 rows x 64 bytes of output
  // row max / row sum exchange of the two warpgroups: [tile parity][max, sum][warpgroup][row]
  static constexpr int XCH_BYTES = NSM == 2 ? 2 * 2 * 2 * 128 * 4 : 0;
  static constexpr int SMEM = 1024 + NPIPE * PIPE_BYTES + NPIPE * PIPE_BARS * 8 + 32 + STG_BYTES + XCH_BYTES;
  static constexpr uint32_t TM_O = 0, TM_S = D, TM_PIPE = 256;
  // threads: softmax warpgroups, the producer / issuer warpgroup and, with
  // two softmax warpgroups on one pipeline, an epilogue warpgroup
  static constexpr int THREADS = NSM == 2 ? 512 : 384;
  static constexpr int REGS_SOFTMAX = NSM == 2 ? 184 : 192, REGS_OTHER = NSM == 2 ? 72 : 120;
  static_assert(2 * REGS_SOFTMAX + (THREADS / 128 - 2) * REGS_OTHER <= 65536 / THREADS * (THREADS / 128),
                "register split");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(NPIPE * (D + 128 * NSM) <= 512, "TMEM columns");
  static_assert(NPIPE * NSM == 2, "two softmax warpgroups");
};
constexpr float kLog2_448 = 8.807354922057604f;  // log2(448)
constexpr float kLn448 = 6.104793232414985f;     // ln(448)

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format code 0),
// both K-major, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four fp32 values -> four E4M3 codes (round to nearest even, saturating to
// +-448), x0 in the lowest byte: consecutive keys of the A operand in TMEM.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

}  // namespace

// First row of sequence b's keys in the transposed V (a multiple of 16):
//   THD: roundup16(cu_kv[b]) + 16b    BSHD: b * roundup16(sk)    SBHD: 0
__device__ __forceinline__ int vt_row0(const Geom& g, int b, const SeqInfo& si) {
  if (g.layout == SDPA_THD) return ((si.krow0 + 15) & ~15) + 16 * b;
  if (g.layout == SDPA_BSHD) return b * ((g.sk + 15) & ~15);
  return 0;
}

// Vt[head][d][vt_row0(b) + key] = V[key row][head][d] for every key of every
// sequence; the rows from the end of a sequence's keys up to the next
// sequence's first row (and up to vt_rows after the last) are zeroed. One
// block per (128-key slice, (kv head, 128-column slice of d), sequence).
__global__ void __launch_bounds__(256) vt_kernel(const Fp8Params p) {
  const Geom& g = p.g;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;
  const int dsl = g.d / 128;
  const int b = blockIdx.z, h = blockIdx.y / dsl, d0 = (blockIdx.y % dsl) * 128, k0 = blockIdx.x * 128;
  const SeqInfo si = seq_info(g, b);
  const int r0 = vt_row0(g, b, si);
  int seg;  // rows of this sequence's segment of Vt (a multiple of 16)
  if (g.layout == SDPA_THD)
    seg = (b + 1 < g.batch ? vt_row0(g, b + 1, seq_info(g, b + 1)) : p.vt_rows) - r0;
  else
    seg = (g.sk + 15) & ~15;
  if (k0 >= seg) return;
  const int kh = si.khead0 + h;
  __shared__ __align__(16) uint8_t t[128][128 + 16];  // [key][d], rows padded against bank conflicts
  for (int it = threadIdx.x; it < 128 * 8; it += 256) {
    const int kk = it >> 3, c = it & 7;
    const int key = k0 + kk;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    const uint8_t* src = p.v + ((long long)(si.krow0 + key) * g.nh_kv + kh) * g.d + d0 + c * 16;
    if (key < si.lk && SDPA_ADDR_OK(g.chk, src, 16)) v = *reinterpret_cast<const uint4*>(src);
    *reinterpret_cast<uint4*>(&t[kk][c * 16]) = v;
  }
  __syncthreads();
  for (int it = threadIdx.x; it < 128 * 8; it += 256) {
    const int d = it >> 3, c = it & 7;
    if (k0 + c * 16 >= seg) continue;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (uint32_t)t[c * 16 + 4 * e][d] | ((uint32_t)t[c * 16 + 4 * e + 1][d] << 8) |
             ((uint32_t)t[c * 16 + 4 * e + 2][d] << 16) | ((uint32_t)t[c * 16 + 4 * e + 3][d] << 24);
    uint8_t* dst = p.vt + ((long long)kh * g.d + d0 + d) * p.vt_rows + r0 + k0 + c * 16;
    if (SDPA_ADDR_OK(g.chk, dst, 16)) *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Key tile (counted from the tile's first) of step k of a pass over n key
// tiles. With two softmax warpgroups taking the steps in turn, the two masked
// edge tiles (the first and the last) go first, one to each warpgroup:
// 0, n - 1, 1, 2, ..., n - 2; with one, in order.
template <int NSM>
__device__ __forceinline__ int key_tile_of(int k, int n) {
  if (NSM == 1 || n < 3) return k;
  return k == 0 ? 0 : (k == 1 ? n - 1 : k - 1);
}

// A query tile of the heaviest-first order (the last query tiles of every
// sequence first, GQA heads adjacent) and the key tiles it sees.
struct Fp8Tile {
  int q0, q_last, t_lo, n, qhead, khead, vrow0;
  SeqInfo si;
  KeyRange kr;
};

__device__ __forceinline__ bool fp8_tile(const Fp8Params& p, int idx, Fp8Tile& t) {
  const Geom& g = p.g;
  const int h = idx % g.hq;
  idx /= g.hq;
  const int b = idx % g.batch;
  idx /= g.batch;
  t.q0 = (p.n_q_tiles - 1 - idx) * F8_BM;
  t.si = seq_info(g, b);
  if (t.q0 >= t.si.lq) return false;
  t.kr = key_range(g, t.si.lq, t.si.lk);
  t.q_last = min(t.q0 + F8_BM - 1, t.si.lq - 1);
  const int lo = t.kr.lo(t.q0), hi = t.kr.hi(t.q_last);
  t.t_lo = lo / F8_BN;
  t.n = hi > lo ? (hi + F8_BN - 1) / F8_BN - t.t_lo : 0;
  t.qhead = t.si.qhead0 + h;
  t.khead = t.si.khead0 + h / (g.hq / g.hkv);
  t.vrow0 = vt_row0(g, b, t.si);
  return true;
}

// Shared-memory objects of one pipeline.
struct Pipe8 {
  uint8_t* sQ;
  uint8_t* sStage;
  uint64_t* full;         // [NST]
  uint64_t* empty;        // [NST]
  uint64_t* bar_q;        // Q of a tile landed
  uint64_t* bar_s;        // [2] S of a step ready, per S buffer
  uint64_t* bar_p;        // [2] the softmax is done with a step (pass 2: P8 written), per S buffer
  uint64_t* bar_o;        // a tile's last P8 V done
  uint64_t* q_free;       // a tile's last S done: Q may be replaced
  uint64_t* o_free;       // the epilogue has read O
  uint64_t* sched_full;   // [2] a tile published
  uint64_t* sched_empty;  // [2] its entry read by the MMA issuer and the softmax warps
  int* sched;             // [2] ticket, or -1 when the work is out
  uint64_t* bar_xm;       // two softmax warpgroups: pass-1 row maxima exchanged
  uint64_t* bar_stats;    // two softmax warpgroups: a tile's row maxima and partial sums in place
};

template <int D>
__device__ __forceinline__ Pipe8 pipe8_at(uint8_t* smem, int x) {
  using C = F8Cfg<D>;
  Pipe8 P;
  P.sQ = smem + x * C::PIPE_BYTES;
  P.sStage = P.sQ + C::TILE;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + C::NPIPE * C::PIPE_BYTES) + x * C::PIPE_BARS;
  P.full = b;
  P.empty = b + C::NST;
  P.bar_q = b + 2 * C::NST;
  P.bar_s = P.bar_q + 1;
  P.bar_p = P.bar_q + 3;
  P.bar_o = P.bar_q + 5;
  P.q_free = P.bar_q + 6;
  P.o_free = P.bar_q + 7;
  P.sched_full = P.bar_q + 8;
  P.sched_empty = P.bar_q + 10;
  P.sched = reinterpret_cast<int*>(P.bar_q + 12);
  P.bar_xm = P.bar_q + 13;
  P.bar_stats = P.bar_q + 14;
  return P;
}

// Columns [32 cc, 32 cc + 32) of one warp's 32 rows of O (row `lane` at TMEM
// lanes ocol) times mul, staged in shared memory (wst, 2 KB; segment k of
// row `lane` at k ^ (lane % 4)) so that each store writes eight rows' 64
// contiguous bytes. Arrives on o_free (if given) once the chunk has been read
// from TMEM.
template <typename E, int D>
__device__ __forceinline__ void store_o_chunk(const Geom& g, uint32_t ocol, int cc, float mul, typename E::T* orow,
                                              bool valid, uint8_t* wst, uint64_t* o_free, int lane) {
  using T = typename E::T;
  uint32_t uu[32];
  tmem_ld32(ocol + cc * 32, uu);
  tmem_wait_ld();
  reg_fence(uu);
  if (o_free) {
    tc_fence_before();
    mbar_arrive(o_free);
  }
  uint32_t packed[16];
#pragma unroll
  for (int k2 = 0; k2 < 16; ++k2)
    packed[k2] = E::pack(__uint_as_float(uu[2 * k2]) * mul, __uint_as_float(uu[2 * k2 + 1]) * mul);
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2)
    *reinterpret_cast<uint4*>(wst + lane * 64 + ((k2 ^ (lane & 3)) << 4)) =
        make_uint4(packed[4 * k2], packed[4 * k2 + 1], packed[4 * k2 + 2], packed[4 * k2 + 3]);
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rr = k * 8 + (lane >> 2), seg = lane & 3;  // row of the warp, 16-byte segment
    const uint4 v4 = *reinterpret_cast<const uint4*>(wst + rr * 64 + ((seg ^ (rr & 3)) << 4));
    T* drow = reinterpret_cast<T*>(__shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(orow), rr));
    const bool vr = __shfl_sync(0xffffffffu, valid ? 1 : 0, rr) != 0;
    if (vr && SDPA_ADDR_OK(g.chk, drow + cc * 32 + seg * 8, 16)) *reinterpret_cast<uint4*>(drow + cc * 32 + seg * 8) = v4;
  }
  __syncwarp();
}

// All D columns of one warp's 32 rows of O, chunk by chunk; o_free after the
// last chunk has been read.
template <typename E, int D>
__device__ __forceinline__ void store_o_rows(const Geom& g, uint32_t ocol, float mul, typename E::T* orow, bool valid,
                                             uint8_t* wst, uint64_t* o_free, int lane) {
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc)
    store_o_chunk<E, D>(g, ocol, cc, mul, orow, valid, wst, cc == D / 32 - 1 ? o_free : nullptr, lane);
}

// A row with no key: O = 0, LSE = -inf.
template <typename T, int D>
__device__ __forceinline__ void store_empty_row(const Geom& g, T* orow, float* lse_at, bool valid) {
  if (valid && SDPA_ADDR_OK(g.chk, orow, 2 * D)) {
    uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
    for (int k2 = 0; k2 < D / 8; ++k2) dst[k2] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (valid && SDPA_ADDR_OK(g.chk, lse_at, 4)) *lse_at = -INFINITY;
}

// Persistent, one CTA per SM. Each pipeline takes query tiles (heaviest
// first) from an atomic ticket counter; a tile runs 2n steps (pass 1 over its
// n key tiles: S and the row max; pass 2: S again, P8 = E4M3(448 P~),
// O += P8 V). Head_dim 128: two pipelines, each step S -> softmax -> (P8 V)
// in turn through the pipeline's single S buffer; the single MMA issuer
// serves the two pipelines strictly in turn, so one pipeline's softmax runs
// while the tensor pipe works on the other's MMAs. Head_dim 256: one
// pipeline, two S buffers, the two softmax warpgroups taking its steps in
// turn. Roles: warps 0-7 softmax + epilogue, warps 8 (/ 9) TMA producer and
// scheduler of pipeline 0 (/ 1), warp 10 TMEM allocator + MMA issuer, warp
// 11 only completes the third warpgroup. Every barrier phase counts across
// tiles.
template <bool BF16, int D>
__global__ void __launch_bounds__(F8Cfg<D>::THREADS, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ Fp8Params p) {
  using E = Elem<BF16>;
  using C = F8Cfg<D>;
  const Geom& g = p.g;
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar_drain = reinterpret_cast<uint64_t*>(smem + C::NPIPE * C::PIPE_BYTES) + C::NPIPE * C::PIPE_BARS;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  uint8_t* stg = reinterpret_cast<uint8_t*>(bar_drain) + 32;  // [8 softmax warps][2 KB] output staging
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int x = 0; x < C::NPIPE; ++x) {
      const Pipe8 P = pipe8_at<D>(smem, x);
      for (int i = 0; i < C::NST; ++i) {
        mbar_init(&P.full[i], 1);
        mbar_init(&P.empty[i], 1);
      }
      mbar_init(P.bar_q, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&P.bar_s[i], 1);
        mbar_init(&P.bar_p[i], 128);
      }
      mbar_init(P.bar_o, 1);
      mbar_init(P.q_free, 1);
      mbar_init(P.o_free, 128);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&P.sched_full[i], 1);
        mbar_init(&P.sched_empty[i], C::NSM == 2 ? 1 + 256 + 128 : 1 + 128);
      }
      mbar_init(P.bar_xm, 256);
      mbar_init(P.bar_stats, 256);
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
    if (warp == 8 || (warp == 9 && C::NPIPE == 2)) {
      // ---------------------------------------------------------- scheduler + producer of pipeline warp - 8
      if (elect_one()) {
        const Pipe8 P = pipe8_at<D>(smem, warp - 8);
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmVt);
        int c = 0, nq = 0, w = 0;
        bool ok = true;
        // the next ticket (a counter the address check rejects hands out none)
        auto take = [&]() {
          return SDPA_ADDR_OK(g.chk, p.tile_counter, 4) ? atomicAdd(p.tile_counter, 1) : p.total_tiles;
        };
        // one ring stage: a K tile (D / 128 boxes of 128 columns) or a Vt tile (one box of D rows)
        auto load = [&](bool vt, int c0, int c1, int c2) -> bool {
          const int slot = c % C::NST;
          if (!mbar_wait(&P.empty[slot], ((c / C::NST) & 1) ^ 1, abort_flag)) return false;
          mbar_arrive_expect_tx(&P.full[slot], C::TILE);
          uint8_t* dst = P.sStage + slot * C::TILE;
          if (vt) {
            tma_load_3d(&tmVt, &P.full[slot], dst, c0, c1, c2);
          } else {
            for (int a = 0; a < C::ATOMS; ++a) tma_load_3d(&tmK, &P.full[slot], dst + a * 16384, c0 + a * 128, c1, c2);
          }
          ++c;
          return true;
        };
        int ticket = take();
        while (true) {
          Fp8Tile t;
          while (ticket < p.total_tiles && !fp8_tile(p, ticket, t)) ticket = take();
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
          mbar_arrive_expect_tx(P.bar_q, C::TILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_3d(&tmQ, P.bar_q, P.sQ + a * 16384, a * 128, t.qhead, t.si.qrow0 + t.q0);
          ++nq;
          // in the order the MMA issuer consumes them (K of step u: key tile
          // u, or u - n in pass 2; Vt of a pass-2 step u: key tile u - n)
          auto load_k = [&](int u) {
            const int j = key_tile_of<C::NSM>(u < t.n ? u : u - t.n, t.n);
            return load(false, 0, t.khead, t.si.krow0 + (t.t_lo + j) * F8_BN);
          };
          auto load_v = [&](int u) {
            return load(true, t.vrow0 + (t.t_lo + key_tile_of<C::NSM>(u - t.n, t.n)) * F8_BN, 0, t.khead);
          };
          if constexpr (C::NSM == 1) {
            // per step: K, then in pass 2 Vt
            for (int u = 0; u < 2 * t.n && ok; ++u) {
              ok = load_k(u);
              if (ok && u >= t.n) ok = load_v(u);
            }
          } else {
            // K of steps 0 and 1; then per step u: Vt in pass 2, K of step u + 2
            ok = load_k(0) && load_k(1);
            for (int u = 0; u < 2 * t.n && ok; ++u) {
              if (u >= t.n) ok = load_v(u);
              if (ok && u + 2 < 2 * t.n) ok = load_k(u + 2);
            }
          }
          if (!ok) break;
        }
        if (!ok) {
          *abort_flag = 1;
          record_error(p.err, SDPA_ERR_TIMEOUT);
        }
        const int first = c > C::NST ? c - C::NST : 0;
        for (int k = first; k < c; ++k) mbar_wait_drain(&P.full[k % C::NST], (k / C::NST) & 1);
        if (nq > 0) mbar_wait_drain(P.bar_q, (nq - 1) & 1);
      }
    } else if (warp == 10) {
      // ---------------------------------------------------------- MMA issuer for both pipelines
      if (C::NSM == 1 && elect_one()) {
        constexpr uint32_t IDESC_S = idesc_e4m3(128, 128), IDESC_O = idesc_e4m3(128, D);
        struct State {
          int w, c, nq, steps, no, n, u;
          bool done;
        };
        State st[2];
        for (int x = 0; x < 2; ++x) st[x] = State{0, 0, 0, 0, 0, 0, 0, x >= C::NPIPE};
        bool ok = true;
        // next tile with keys of pipeline x (false: its work is out, or a wait failed)
        auto next_item = [&](int x) -> bool {
          const Pipe8 P = pipe8_at<D>(smem, x);
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
            Fp8Tile t;
            fp8_tile(p, item, t);
            if (t.n == 0) continue;
            if (!mbar_wait(P.bar_q, m.nq & 1, abort_flag)) {
              ok = false;
              return false;
            }
            ++m.nq;
            tc_fence_after();
            m.n = t.n;
            m.u = 0;
            return true;
          }
        };
        // S of step u of pipeline x (its previous step's P8 V has been issued,
        // so P8 in the S buffer is consumed first)
        auto issue_s = [&](int x) -> bool {
          const Pipe8 P = pipe8_at<D>(smem, x);
          State& m = st[x];
          const int slot = m.c % C::NST;
          if (!mbar_wait(&P.full[slot], (m.c / C::NST) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t q_base = smem_u32(P.sQ), kb = smem_u32(P.sStage + slot * C::TILE);
#pragma unroll
          for (int ks = 0; ks < D / 32; ++ks) {  // 32 one-byte columns per MMA, four per 128-column atom
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            mma_f8_ss(tmem + x * C::TM_PIPE + C::TM_S, smem_desc_sw128(q_base + off, 16, 1024),
                      smem_desc_sw128(kb + off, 16, 1024), IDESC_S, ks != 0);
          }
          mma_commit(&P.empty[slot]);
          if (m.u == 2 * m.n - 1) mma_commit(P.q_free);
          mma_commit(&P.bar_s[0]);
          ++m.c;
          return true;
        };
        // once the softmax is done with step u: in pass 2, O += P8 V (the
        // tile's first P8 V overwrites O, which the previous tile's epilogue
        // must have read)
        auto after_softmax = [&](int x) -> bool {
          const Pipe8 P = pipe8_at<D>(smem, x);
          State& m = st[x];
          if (m.u == m.n && m.no > 0 && !mbar_wait(P.o_free, (m.no - 1) & 1, abort_flag)) return false;
          if (!mbar_wait(&P.bar_p[0], m.steps & 1, abort_flag)) return false;
          ++m.steps;
          if (m.u < m.n) return true;  // pass 1: the max only
          const int slot = m.c % C::NST;
          if (!mbar_wait(&P.full[slot], (m.c / C::NST) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t vb = smem_u32(P.sStage + slot * C::TILE);
          const uint32_t pcol = tmem + x * C::TM_PIPE + C::TM_S;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // 32 keys per MMA: 8 TMEM columns of packed P8; N = D rows of Vt
            mma_f8_ts(tmem + x * C::TM_PIPE + C::TM_O, pcol + ks * 8, smem_desc_sw128(vb + ks * 32, 16, 1024),
                      IDESC_O, (m.u - m.n) > 0 || ks != 0);
          mma_commit(&P.empty[slot]);
          ++m.c;
          return true;
        };
        for (int x = 0; x < C::NPIPE && ok; ++x)
          if (next_item(x) && !issue_s(x)) ok = false;
        while (ok && !(st[0].done && st[1].done)) {
          for (int x = 0; x < 2 && ok; ++x) {
            State& m = st[x];
            if (m.done) continue;
            if (!after_softmax(x)) {
              ok = false;
              break;
            }
            if (m.u == 2 * m.n - 1) {
              mma_commit(pipe8_at<D>(smem, x).bar_o);
              ++m.no;
              if (!next_item(x)) continue;  // out of work (or ok cleared)
            } else {
              ++m.u;
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
      } else if (C::NSM == 2 && elect_one()) {
        // ---- one pipeline, two S buffers: step u of a tile runs in buffer
        // u % 2 and on softmax warpgroup u % 2. Per tile: S of steps 0 and 1,
        // then for each step u once its softmax is done: P8 V (pass 2) and S
        // of step u + 2 into the buffer just freed, so the tensor pipe works
        // on the next steps while the other warpgroup's softmax runs.
        constexpr uint32_t IDESC_S = idesc_e4m3(128, 128), IDESC_O = idesc_e4m3(128, D);
        const Pipe8 P = pipe8_at<D>(smem, 0);
        int w = 0, c = 0, nq = 0, no = 0;
        int base = 0;  // steps each S buffer served in earlier tiles (n per tile)
        bool ok = true;
        auto issue_s = [&](int u, int n) -> bool {
          const int slot = c % C::NST;
          if (!mbar_wait(&P.full[slot], (c / C::NST) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t q_base = smem_u32(P.sQ), kb = smem_u32(P.sStage + slot * C::TILE);
          const uint32_t dcol = tmem + C::TM_S + (uint32_t)(u & 1) * 128;
#pragma unroll
          for (int ks = 0; ks < D / 32; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            mma_f8_ss(dcol, smem_desc_sw128(q_base + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024), IDESC_S,
                      ks != 0);
          }
          mma_commit(&P.empty[slot]);
          if (u == 2 * n - 1) mma_commit(P.q_free);
          mma_commit(&P.bar_s[u & 1]);
          ++c;
          return true;
        };
        // the tile's first P8 V overwrites O, which the previous tile's
        // epilogue must have read
        auto issue_pv = [&](int u, int n) -> bool {
          if (u == n && no > 0 && !mbar_wait(P.o_free, (no - 1) & 1, abort_flag)) return false;
          const int slot = c % C::NST;
          if (!mbar_wait(&P.full[slot], (c / C::NST) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t vb = smem_u32(P.sStage + slot * C::TILE);
          const uint32_t pcol = tmem + C::TM_S + (uint32_t)(u & 1) * 128;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_f8_ts(tmem + C::TM_O, pcol + ks * 8, smem_desc_sw128(vb + ks * 32, 16, 1024), IDESC_O,
                      u > n || ks != 0);
          mma_commit(&P.empty[slot]);
          ++c;
          return true;
        };
        while (ok) {
          const int e = w & 1;
          if (!mbar_wait(&P.sched_full[e], (w >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const int item = *reinterpret_cast<volatile int*>(&P.sched[e]);
          mbar_arrive(&P.sched_empty[e]);
          ++w;
          if (item < 0) break;
          Fp8Tile t;
          fp8_tile(p, item, t);
          const int n = t.n;
          if (n == 0) continue;
          if (!mbar_wait(P.bar_q, nq & 1, abort_flag)) {
            ok = false;
            break;
          }
          ++nq;
          tc_fence_after();
          ok = issue_s(0, n) && issue_s(1, n);
          for (int u = 0; u < 2 * n && ok; ++u) {
            ok = mbar_wait(&P.bar_p[u & 1], (base + (u >> 1)) & 1, abort_flag);
            if (ok && u >= n) ok = issue_pv(u, n);
            if (ok && u + 2 < 2 * n) ok = issue_s(u + 2, n);
          }
          if (!ok) break;
          base += n;
          mma_commit(P.bar_o);
          ++no;
        }
        if (!ok) {
          *abort_flag = 1;
          record_error(p.err, SDPA_ERR_TIMEOUT);
          mma_commit(bar_drain);
          mbar_wait_drain(bar_drain, 0);
        }
      }
    } else if (C::NSM == 2 && warp >= 12) {
      // ---------------------------------------------------------- epilogue warpgroup (two softmax warpgroups)
      // Per tile: the row's max and sum from the two softmax warpgroups'
      // stats, then O / the row sum from TMEM and the LSE; the softmax
      // warpgroups meanwhile run the next tile's pass 1. Its tile-queue entry
      // is released only after the stats are read, so no stats slot is
      // rewritten (by the tile after next) before that.
      using T = typename E::T;
      const Pipe8 P = pipe8_at<D>(smem, 0);
      const int r = (warp & 3) * 32 + lane;
      const uint32_t ocol = tmem + C::TM_O + ((uint32_t)((warp & 3) * 32) << 16);
      const float* xch = reinterpret_cast<const float*>(stg + C::STG_BYTES);
      int w = 0, no = 0;
      bool ok = true;
      while (ok) {
        const int e = w & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&P.sched_full[e], (w >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        const int item = *reinterpret_cast<volatile int*>(&P.sched[e]);
        ++w;
        if (item < 0) {
          mbar_arrive(&P.sched_empty[e]);
          break;
        }
        Fp8Tile t;
        fp8_tile(p, item, t);
        const int i = t.q0 + r;
        const bool valid = i < t.si.lq;
        T* orow = reinterpret_cast<T*>(p.o) + ((long long)(t.si.qrow0 + i) * g.nh_q + t.qhead) * D;
        float* lse_at = p.lse + (long long)(t.si.qrow0 + i) * g.nh_q + t.qhead;
        if (t.n == 0) {
          mbar_arrive(&P.sched_empty[e]);
          store_empty_row<T, D>(g, orow, lse_at, valid);
          continue;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(P.bar_stats, no & 1, abort_flag))) {
          ok = false;
          break;
        }
        const float* xs = xch + (no & 1) * 512;
        const float m = fmaxf(xs[r], xs[128 + r]), l = xs[256 + r] + xs[384 + r];
        mbar_arrive(&P.sched_empty[e]);
        if (!__all_sync(0xffffffffu, mbar_wait(P.bar_o, no & 1, abort_flag))) {
          ok = false;
          break;
        }
        ++no;
        tc_fence_after();
        const float mul = l > 0.f ? p.o_scale * 448.f / l : 0.f;  // o_scale = d_v / 448
        store_o_rows<E, D>(g, ocol, mul, orow, valid, stg + (warp - 12) * 2048, P.o_free, lane);
        if (valid && SDPA_ADDR_OK(g.chk, lse_at, 4))
          *lse_at = l > 0.f ? m * g.scale + (logf(l) - kLn448) : -INFINITY;
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
    }
  } else {
    regs_inc<C::REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax + epilogue
    // head_dim 128: warpgroup wg serves pipeline wg, every step of its tiles.
    // head_dim 256: both serve the one pipeline, warpgroup wg the steps u with
    // u % 2 == wg in S buffer wg; they exchange the pass-1 row maxima before
    // pass 2 and the row sums before the epilogue, and each stores half of O.
    const int wg = warp >> 2;
    const int x = C::NSM == 2 ? 0 : wg, sb = C::NSM == 2 ? wg : 0;
    {
      const Pipe8 P = pipe8_at<D>(smem, x);
      const int r = (warp & 3) * 32 + lane;
      const uint32_t lane_base = tmem + x * C::TM_PIPE + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t scol = lane_base + C::TM_S + (uint32_t)sb * 128;
      float* xch = reinterpret_cast<float*>(stg + C::STG_BYTES);  // [tile parity][max, sum][warpgroup][row]
      const float sl2 = g.scale_log2;
      using T = typename E::T;
      int w = 0, steps = 0, no = 0, xt = 0;
      bool ok = true;
      // head_dim 128: a finished tile's O is stored one 32-column chunk per
      // pass-1 step of the pipeline's next tile (pass 1 does not touch O), the
      // rest before its first pass-2 step (whose P8 V needs o_free)
      int pend = 0;  // chunks of the previous tile's O still to store
      bool pneed_o = false;
      float pmul = 0.f;
      T* porow = nullptr;
      bool pvalid = false;
      auto drain_one = [&]() -> bool {
        if (pneed_o) {  // that tile's last P8 V is done (this keeps every bar_o phase waited in turn)
          if (!__all_sync(0xffffffffu, mbar_wait(P.bar_o, no & 1, abort_flag))) return false;
          ++no;
          tc_fence_after();
          pneed_o = false;
        }
        store_o_chunk<E, D>(g, lane_base + C::TM_O, D / 32 - pend, pmul, porow, pvalid, stg + warp * 2048,
                            pend == 1 ? P.o_free : nullptr, lane);
        --pend;
        return true;
      };
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
        Fp8Tile t;
        fp8_tile(p, item, t);
        const int n = t.n;
        const int i = t.q0 + r;
        const bool valid = i < t.si.lq;
        const int lo_i = t.kr.lo(i), hi_i = t.kr.hi(i);
        const int lo_last = t.kr.lo(t.q_last), hi_first = t.kr.hi(t.q0);
        T* orow = reinterpret_cast<T*>(p.o) + ((long long)(t.si.qrow0 + i) * g.nh_q + t.qhead) * D;
        float* lse_at = p.lse + (long long)(t.si.qrow0 + i) * g.nh_q + t.qhead;
        if (n == 0) {  // no key for any row of the tile (the epilogue warpgroup's, if there is one)
          if (C::NSM == 1) store_empty_row<T, D>(g, orow, lse_at, valid);
          continue;
        }
        // pass 1: the row max, four independent chains; pass 2: the exponent's
        // bias log2(448) - m * scale * log2e, so exp2 gives 448 P~ directly,
        // and the sum of 448 P~ (two lanes)
        float mm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float m = -INFINITY, nb = 0.f;
        float2 l2 = make_float2(0.f, 0.f);
        bool have_m = false;
        // the row max once pass 1 is done (with two warpgroups: the larger of
        // the two partial maxima) and the exponent's bias from it
        auto final_max = [&]() -> bool {
          m = fmaxf(fmaxf(mm[0], mm[1]), fmaxf(mm[2], mm[3]));
          if constexpr (C::NSM == 2) {
            float* xm = xch + (xt & 1) * 512;
            xm[wg * 128 + r] = m;
            mbar_arrive(P.bar_xm);
            if (!__all_sync(0xffffffffu, mbar_wait(P.bar_xm, xt & 1, abort_flag))) return false;
            m = fmaxf(m, xm[(1 - wg) * 128 + r]);
          }
          nb = kLog2_448 - (m == -INFINITY ? 0.f : m * sl2);
          have_m = true;
          return true;
        };
        for (int u = sb; u < 2 * n; u += C::NSM) {
          if (u >= n && !have_m && !final_max()) {
            ok = false;
            break;
          }
          if (C::NSM == 1 && u == n) {
            while (pend > 0 && ok) ok = drain_one();
            if (!ok) break;
          }
          if (!__all_sync(0xffffffffu, mbar_wait(&P.bar_s[sb], steps & 1, abort_flag))) {
            ok = false;
            break;
          }
          ++steps;
          tc_fence_after();
          const int kb = (t.t_lo + key_tile_of<C::NSM>(u < n ? u : u - n, n)) * F8_BN;
          const bool edge = !(lo_last <= kb && hi_first >= kb + F8_BN);  // uniform across the tile
          if (u < n && !edge) {
            // interior pass-1 step: the row max comes with the loads
            uint32_t u0[32], u1[32], u2[32], u3[32];
            float x0, x1, x2, x3;
            tmem_ld32_max(scol, u0, x0);
            tmem_ld32_max(scol + 32, u1, x1);
            tmem_ld32_max(scol + 64, u2, x2);
            tmem_ld32_max(scol + 96, u3, x3);
            tmem_wait_ld();
            asm volatile("" : "+f"(x0), "+f"(x1), "+f"(x2), "+f"(x3));
            mm[0] = fmaxf(mm[0], x0);
            mm[1] = fmaxf(mm[1], x1);
            mm[2] = fmaxf(mm[2], x2);
            mm[3] = fmaxf(mm[3], x3);
          } else {
            float s[128];
            {
              uint32_t u0[32], u1[32], u2[32], u3[32];
              tmem_ld32(scol, u0);
              tmem_ld32(scol + 32, u1);
              tmem_ld32(scol + 64, u2);
              tmem_ld32(scol + 96, u3);
              tmem_wait_ld();
              reg_fence(u0);
              reg_fence(u1);
              reg_fence(u2);
              reg_fence(u3);
#pragma unroll
              for (int cc = 0; cc < 32; ++cc) {
                s[cc] = __uint_as_float(u0[cc]);
                s[32 + cc] = __uint_as_float(u1[cc]);
                s[64 + cc] = __uint_as_float(u2[cc]);
                s[96 + cc] = __uint_as_float(u3[cc]);
              }
            }
            if (edge) {
#pragma unroll
              for (int cc = 0; cc < 128; ++cc) s[cc] = in_range(kb + cc, lo_i, hi_i) ? s[cc] : -INFINITY;
            }
            if (u < n) {
#pragma unroll
              for (int cc = 0; cc < 128; ++cc) mm[cc & 3] = fmaxf(mm[cc & 3], s[cc]);
            } else {
              uint32_t pk[32];
              const float2 sc2 = make_float2(sl2, sl2), nb2 = make_float2(nb, nb);
              float2 ra = make_float2(0.f, 0.f), rb = make_float2(0.f, 0.f);
#pragma unroll
              for (int cc = 0; cc < 32; ++cc) {
                const float2 ta = ffma2(make_float2(s[4 * cc], s[4 * cc + 1]), sc2, nb2);
                const float2 tb = ffma2(make_float2(s[4 * cc + 2], s[4 * cc + 3]), sc2, nb2);
                const float2 pa = make_float2(ex2(ta.x), ex2(ta.y)), pb = make_float2(ex2(tb.x), ex2(tb.y));
                ra = fadd2(ra, pa);
                rb = fadd2(rb, pb);
                pk[cc] = pack_e4m3x4(pa.x, pa.y, pb.x, pb.y);  // 448 P~, rounded once to E4M3
              }
              l2 = fadd2(l2, fadd2(ra, rb));
              tmem_st32(scol, pk);  // P8 into the S buffer's first 32 columns
              tmem_wait_st();
            }
          }
          tc_fence_before();
          mbar_arrive(&P.bar_p[sb]);
          if (C::NSM == 1 && u < n && pend > 0 && !drain_one()) {
            ok = false;
            break;
          }
        }
        if (ok && !have_m && !final_max()) ok = false;  // a warpgroup with no pass-2 step
        if (!ok) break;
        const float l = l2.x + l2.y;  // the sum of 448 P~ over this warpgroup's steps
        if constexpr (C::NSM == 2) {
          // the partial sum beside the maxima, for the epilogue warpgroup
          xch[(xt & 1) * 512 + 256 + wg * 128 + r] = l;
          mbar_arrive(P.bar_stats);
          ++xt;
        } else {
          // the LSE now; O / the row sum during the pipeline's next tile
          if (valid && SDPA_ADDR_OK(g.chk, lse_at, 4))
            *lse_at = l > 0.f ? m * g.scale + (logf(l) - kLn448) : -INFINITY;
          pend = D / 32;
          pneed_o = true;
          pmul = l > 0.f ? p.o_scale * 448.f / l : 0.f;  // o_scale = d_v / 448
          porow = orow;
          pvalid = valid;
        }
      }
      while (ok && pend > 0) ok = drain_one();  // the pipeline's last tile
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, SDPA_ERR_TIMEOUT);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int launch_vt(const Fp8Params& p, cudaStream_t stream) {
  const int max_seg = p.g.layout == SDPA_THD ? p.g.sk + 32 : ((p.g.sk + 15) & ~15);
  if (p.g.batch <= 0 || max_seg <= 0) return SDPA_OK;
  if (p.g.batch > 65535 || p.g.hkv > 65535) return SDPA_ERR_UNSUPPORTED;
  if ((long long)p.g.hkv * (p.g.d / 128) > 65535) return SDPA_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)((max_seg + 127) / 128), (unsigned)(p.g.hkv * (p.g.d / 128)), (unsigned)p.g.batch);
  vt_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

template <bool BF16, int D>
static int launch_fwd_fp8_t(const Fp8Launch& L, long long tiles) {
  using C = F8Cfg<D>;
  auto kern = fwd_fp8_kernel<BF16, D>;
  if (const int rc = set_kernel_smem(reinterpret_cast<const void*>(kern), C::SMEM, 100)) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDPA_ERR_CUDA;
  Fp8Params p = L.p;
  p.total_tiles = (int)tiles;
  long long grid = std::min<long long>((tiles + C::NPIPE - 1) / C::NPIPE, sms);
  if (debug_max_ctas() > 0) grid = std::min<long long>(grid, debug_max_ctas());  // tickets cover every tile
  if (cudaMemsetAsync(p.tile_counter, 0, sizeof(int), L.stream) != cudaSuccess) return SDPA_ERR_CUDA;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, L.stream>>>(L.tmQ, L.tmK, L.tmVt, p);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

int launch_fwd_fp8(const Fp8Launch& L, bool bf16) {
  const long long tiles = (long long)L.p.n_q_tiles * L.p.g.hq * L.p.g.batch;
  if (tiles <= 0) return SDPA_OK;
  if (tiles > 0x7fffffffLL - 4096) return SDPA_ERR_UNSUPPORTED;
  if (L.p.g.d == 128) return bf16 ? launch_fwd_fp8_t<true, 128>(L, tiles) : launch_fwd_fp8_t<false, 128>(L, tiles);
  if (L.p.g.d == 256) return bf16 ? launch_fwd_fp8_t<true, 256>(L, tiles) : launch_fwd_fp8_t<false, 256>(L, tiles);
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace sdpa
