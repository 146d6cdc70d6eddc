// common.cuh -- geometry shared by the kernels: the generic "rows x heads x D"
// view of every layout, per-sequence bounds, and the mask/window ranges.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/sdpa.h"

namespace sdpa {

// Every layout is addressed as x[row][head][d] with
//   BSHD: row = b*S + s, head = h           (rows = B*S, heads = H)
//   SBHD: row = s,       head = b*H + h     (rows = S,   heads = B*H)
//   THD:  row = cu[b]+s, head = h           (rows = T,   heads = H)
// so one 3-D TMA tensor map {D, heads, rows} serves all three, and the
// token-major LSE index is row*heads + head.
// Extents of the buffers one call was given, for the address-checked build
// (SDPA_ADDR_CHECK; see addr_ok). One table per device, in device memory.
constexpr int kAddrExtents = 16;
struct AddrTable {
  unsigned long long n;                                   // extents in use
  unsigned long long lo[kAddrExtents], hi[kAddrExtents];  // [lo, hi) byte ranges
  int* err;                                               // the device error word
  unsigned long long violations, first_addr, first_bytes;
};

struct Geom {
  int layout, mask, batch, sq, sk;  // THD: sq/sk are the largest lengths
  int hq, hkv, d;
  int dv;  // width of V and O rows (== d except for the asymmetric forward)
  int wl, wr;  // window; wr == 0 for causal masks, < 0 = unbounded
  float scale, scale_log2;
  int rows_q, rows_kv;  // rows of the generic view
  int nh_q, nh_kv;      // heads of the generic view
  const int32_t* cu_q;
  const int32_t* cu_kv;
  AddrTable* chk;  // address-checked build: this call's extents; else null
};

// Address check of a load or store at a computed global address (every access
// that is not a tensor-map copy, which the hardware bounds against its map).
// The checked build tests [p, p + bytes) against the call's extents; outside
// all of them the access is to be skipped: the violation is counted, its
// address kept and SDPA_ERR_ADDRESS recorded. Elsewhere the test is `true`.
#ifdef SDPA_ADDR_CHECK
static __device__ __forceinline__ bool addr_ok(AddrTable* t, const void* p, unsigned long long bytes) {
  if (!t) return true;
  const unsigned long long a = reinterpret_cast<unsigned long long>(p);
  const unsigned long long n = t->n < (unsigned long long)kAddrExtents ? t->n : kAddrExtents;
  for (unsigned long long i = 0; i < n; ++i)
    if (a >= t->lo[i] && bytes <= t->hi[i] - t->lo[i] && a - t->lo[i] <= t->hi[i] - t->lo[i] - bytes) return true;
  if (atomicAdd(&t->violations, 1ull) == 0ull) {
    t->first_addr = a;
    t->first_bytes = bytes;
  }
  if (t->err) atomicCAS(t->err, 0, (int)SDPA_ERR_ADDRESS);
  return false;
}
#define SDPA_ADDR_OK(t, p, bytes) ::sdpa::addr_ok((t), (p), (unsigned long long)(bytes))
#else
#define SDPA_ADDR_OK(t, p, bytes) true
#endif

// Per-row backward statistics (-LSE*log2e and delta) are stored per generic
// head as [head][stat_rows]; query s of sequence b sits at srow0 + s. Every
// sequence starts on a multiple of four rows (16 bytes), so a 64-row query
// tile's statistics are one aligned block that bulk copies and vector loads
// can take as it is:
//   THD:  roundup4(cu_q[b]) + 4b     BSHD: b * roundup4(sq)     SBHD: 0
// (SBHD keeps batches apart through the generic head.)
struct SeqInfo {
  int lq, lk;          // lengths of this sequence
  int qrow0, krow0;    // first generic row
  int qhead0, khead0;  // generic head offset
  int srow0;           // row of query 0 in the backward statistics arrays
};

__device__ __forceinline__ SeqInfo seq_info(const Geom& g, int b) {
  SeqInfo s;
  if (g.layout == SDPA_THD) {
    if (!SDPA_ADDR_OK(g.chk, g.cu_q + b, 8) || !SDPA_ADDR_OK(g.chk, g.cu_kv + b, 8)) {
      s.qrow0 = s.krow0 = s.lq = s.lk = s.qhead0 = s.khead0 = s.srow0 = 0;  // an empty sequence
      return s;
    }
    s.qrow0 = g.cu_q[b];
    s.lq = g.cu_q[b + 1] - s.qrow0;
    s.krow0 = g.cu_kv[b];
    s.lk = g.cu_kv[b + 1] - s.krow0;
    s.qhead0 = s.khead0 = 0;
    s.srow0 = ((s.qrow0 + 3) & ~3) + 4 * b;
  } else if (g.layout == SDPA_BSHD) {
    s.lq = g.sq;
    s.lk = g.sk;
    s.qrow0 = b * g.sq;
    s.krow0 = b * g.sk;
    s.qhead0 = s.khead0 = 0;
    s.srow0 = b * ((g.sq + 3) & ~3);
  } else {
    s.lq = g.sq;
    s.lk = g.sk;
    s.qrow0 = s.krow0 = 0;
    s.qhead0 = b * g.hq;
    s.khead0 = b * g.hkv;
    s.srow0 = 0;
  }
  return s;
}

// Keys allowed for query i of a sequence with lengths (lq, lk): [lo, hi).
// The diagonal of row i is key i (top-left, and no-mask windows) or
// i + lk - lq (bottom-right).
struct KeyRange {
  int off, wl, wr, lk;
  __device__ __forceinline__ int lo(int i) const { return wl >= 0 ? max(0, i + off - wl) : 0; }
  __device__ __forceinline__ int hi(int i) const { return wr >= 0 ? min(lk, max(0, i + off + wr + 1)) : lk; }
};

__device__ __forceinline__ KeyRange key_range(const Geom& g, int lq, int lk) {
  KeyRange r;
  r.off = (g.mask == SDPA_MASK_CAUSAL_BOTTOM_RIGHT) ? lk - lq : 0;
  r.wl = g.wl;
  r.wr = g.wr;
  r.lk = lk;
  return r;
}

// Queries that may attend key j: [qlo, qhi) (the inverse of KeyRange).
__device__ __forceinline__ int query_lo(const KeyRange& r, int j) { return r.wr >= 0 ? max(0, j - r.off - r.wr) : 0; }
__device__ __forceinline__ int query_hi(const KeyRange& r, int j, int lq) {
  return r.wl >= 0 ? min(lq, max(0, j - r.off + r.wl + 1)) : lq;
}

// key in [lo, hi) as one unsigned compare, so masking compiles to a select
// rather than a branch per element (an empty range, hi <= lo, admits nothing).
__device__ __forceinline__ bool in_range(int key, int lo, int hi) {
  return (unsigned)(key - lo) < (unsigned)max(hi - lo, 0);
}

template <bool BF16>
struct Elem;
template <>
struct Elem<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
  }
};
template <>
struct Elem<false> {
  using T = __half;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    __half2 v = *reinterpret_cast<__half2*>(&u);
    return __half22float2(v);
  }
};

// Record `code` in the device error word unless an error is already there.
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

}  // namespace sdpa
