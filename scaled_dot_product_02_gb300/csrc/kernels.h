// kernels.h -- parameter blocks and launchers shared between the C-ABI layer
// (api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace sdpa {

// Testing aid (sdpa_debug_set_max_ctas): the most CTAs a kernel may have in
// one launch, 0 = no cap.
int debug_max_ctas();

// Launch `total` CTAs as one grid, or, under a CTA cap, as successive grids of
// at most that many CTAs: fn(offset, count) launches CTAs [offset,
// offset + count) of the index space (kernels add their params' item_offset
// to blockIdx.x). Returns the first failing status.
template <class F>
int launch_in_grids(long long total, F&& fn) {
  const long long cap = debug_max_ctas();
  if (cap <= 0 || total <= cap) return total > 0 ? fn(0LL, total) : 0;
  for (long long off = 0; off < total; off += cap) {
    const int rc = fn(off, total - off < cap ? total - off : cap);
    if (rc) return rc;
  }
  return 0;
}

// Raise a kernel's dynamic shared-memory limit to `bytes` and, when
// carveout >= 0, set its preferred shared-memory carveout (percent), once per
// (kernel, current device): function attributes belong to each device's
// instance of the module, and several host threads may make their first call
// at the same time. Returns an sdpa_status.
int set_kernel_smem(const void* kernel, int bytes, int carveout);
// Device address of a __device__ variable (its host-side stand-in `symbol`)
// on the current device, cached per device for the context it was taken in: a
// context created later (after cudaDeviceReset) looks the address up again.
// nullptr on failure.
void* device_symbol_address(const void* symbol);

struct FwdParams {
  Geom g;
  void* o;
  float* lse;
  int* err;          // sticky per-device error word
  const int* guard;  // per-call metadata-guard result (THD) or nullptr
  int n_q_tiles;     // ceil(seqlen_q / 128)
  int dv_splits;     // 1, or 2 when each CTA owns half of the value columns
  int* tile_counter;  // head_dim 128: ticket counter in the workspace (zeroed per call)
  int total_tiles;    // head_dim 128: tickets (query tiles x heads x batch)
  int item_offset;       // added to blockIdx.x (launches split under a CTA cap)
};

struct FwdLaunch {
  CUtensorMap tmQ, tmK, tmV;
  FwdParams p;
  cudaStream_t stream;
};

int launch_fwd(const FwdLaunch& L, int head_dim, int head_dim_v, bool bf16);

struct BwdParams {
  Geom g;
  float* dq_acc;         // [nh_q][rows_q][D] fp32, zeroed by the preprocess kernel
  const float* lse2;     // [nh_q][stat_rows] -LSE * log2(e) (-inf for rows without keys)
  const float* delta;    // [nh_q][stat_rows] rowsum(dO * O)
  int stat_rows;         // padded row count of lse2/delta (>= rows_q + 64, multiple of 4)
  void* dk;
  void* dv;
  int* err;
  const int* guard;
  int n_kv_tiles;        // ceil(seqlen_kv / 128)
  int d_lo, d_hi;        // dK/dV columns this launch owns (all of D for head_dim 128)
  int item_offset;       // added to blockIdx.x (launches split under a CTA cap)
  const int* order;      // THD: sequence indices, longest first (written by the guard); else null
  int head_block;        // kv heads whose key tiles interleave in the grid (divides hkv)
};

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmDO;
  BwdParams p;
  cudaStream_t stream;
};

// with_dq = false: dK and dV only (the deterministic backward forms dQ with
// launch_dq128 instead of fp32 reductions).
int launch_bwd_dkdv(const BwdLaunch& L, int head_dim, bool bf16, bool with_dq, int* launches);

// Deterministic head_dim 128 dQ (bwd_dq.cu): per query tile, key tiles in a
// fixed order, dQ accumulated in TMEM and written once.
struct DqParams {
  Geom g;
  void* dq;             // written (dtype, scaled)
  const float* nlse2;   // [nh_q][stat_rows] -LSE * log2(e)
  const float* delta;   // [nh_q][stat_rows]
  int stat_rows;
  int* err;
  const int* guard;
  int n_q_tiles;
  int item_offset;       // added to blockIdx.x (launches split under a CTA cap)
};
struct DqLaunch {
  CUtensorMap tmQ, tmDO, tmK, tmV;  // 128-row boxes
  DqParams p;
  cudaStream_t stream;
};
int launch_dq128(const DqLaunch& L, bool bf16);

// head_dim 256/512 backward (bwd_big.cu): score kernels write 16-bit P and
// dS tiles, GEMM kernels form dQ, dV, dK from them.
struct BigBwdParams {
  Geom g;
  uint8_t* p_tiles;      // [B][Hq][n_q_tiles][slots] 32 KB tile images of one key-tile chunk
  uint8_t* ds_tiles;     // same shape
  const float* nlse2;    // [nh_q][stat_rows] -LSE * log2(e)
  const float* delta;    // [nh_q][stat_rows]
  int stat_rows;
  void* dq;
  void* dk;
  void* dv;
  int* err;
  const int* guard;
  int n_q_tiles, n_kv_tiles, slots;
  int chunk_lo, chunk_hi;  // key tiles [chunk_lo, chunk_hi) of this launch set
  int chunk;               // key tiles per chunk (the last chunk may be shorter)
  float* dq_acc;           // [nh_q][rows_q][D] fp32 dQ sum over chunks, zeroed by the
                           // preprocess; nullptr when one chunk covers every key tile
  int item_offset;       // added to blockIdx.x (launches split under a CTA cap)
  int block_major;       // phase-2 grid by (batch, kv head) block (bounded window) or by mode
};

struct BigBwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmDO;    // 128-row boxes
  CUtensorMap tmQ64, tmK64, tmDO64;    // 64-row boxes
  BigBwdParams p;
  cudaStream_t stream;
};

int launch_bwd_big(const BigBwdLaunch& L, int head_dim, bool bf16, int* launches);

// FP8 E4M3 forward, head_dim 128 (fwd_fp8.cu): vt_kernel writes V transposed
// into the workspace, fwd_fp8_kernel computes O and LSE.
struct Fp8Params {
  Geom g;               // scale / scale_log2 include the Q and K descales
  const uint8_t* v;     // E4M3 V [rows_kv][nh_kv][128]
  uint8_t* vt;          // transposed V [nh_kv][128][vt_rows] (workspace)
  int vt_rows;          // keys of Vt per (head, d): every sequence 16-aligned, gaps zero
  void* o;              // [rows_q][nh_q][128], bf16 or fp16
  float* lse;
  int* err;
  const int* guard;
  int n_q_tiles;
  float o_scale;        // d_v / 448 (the epilogue divides by the row sum as well)
  int total_tiles;      // query tiles of the order (tickets of the persistent forward)
  int* tile_counter;    // ticket counter in the workspace (zeroed per call)
};
struct Fp8Launch {
  CUtensorMap tmQ, tmK, tmVt;  // E4M3 128-byte rows, 128-row boxes; Vt 128 keys x 128 d boxes
  Fp8Params p;
  cudaStream_t stream;
};
int launch_vt(const Fp8Params& p, cudaStream_t stream);
int launch_fwd_fp8(const Fp8Launch& L, bool bf16);

// Memory-bound helpers (aux.cu).
struct PrepParams {
  Geom g;
  const void* o;
  const void* dout;
  const float* lse;
  float* lse2;
  float* delta;
  int stat_rows;
  float* dq_acc;  // zeroed here when non-null
  const int* guard;
};
// order (THD backward, else null): receives the sequence indices, longest first
int launch_guard(const Geom& g, int total_q, int total_kv, int* guard, int* err, cudaStream_t s,
                 int* order = nullptr);
int launch_preprocess(const PrepParams& pp, bool bf16, cudaStream_t s);
int launch_wait_selftest(uint64_t limit_ns, int* err, cudaStream_t s);
int launch_dq_finalize(const Geom& g, const float* dq_acc, void* dq, const int* guard, bool bf16, cudaStream_t s);

// Log-sum-exp merge of partial results over a split of the keys (merge.cu).
int launch_merge(const void* o_parts, const float* lse_parts, void* o, float* lse, long long items, int head_dim,
                 int n_parts, bool bf16, AddrTable* chk, cudaStream_t s);

}  // namespace sdpa
