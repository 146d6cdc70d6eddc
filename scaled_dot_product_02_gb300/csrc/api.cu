// api.cu -- the C ABI declared in include/sdpa.h: host-side validation,
// TMA descriptor encoding, workspace carving and kernel launches. No call
// here allocates device memory or synchronises, except
// sdpa_get_device_error, which is documented to synchronise.
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "../../include/sdpa.h"
#include "kernels.h"

// The per-device error word. Kernels receive its device address.
static __device__ int g_sdpa_error_word;

namespace sdpa {
namespace {

thread_local int t_last_launches = 0;

// Event pairs recorded around launches while profiling is on (this thread).
struct Profiler {
  bool on = false;
  struct Mark {
    cudaEvent_t a, b;
    int kind;
  };
  std::vector<Mark> marks;
  size_t used = 0;
  Mark* next(int kind) {
    if (!on || used >= 65536) return nullptr;
    if (used == marks.size()) {
      Mark m{nullptr, nullptr, kind};
      if (cudaEventCreate(&m.a) != cudaSuccess || cudaEventCreate(&m.b) != cudaSuccess) return nullptr;
      marks.push_back(m);
    }
    Mark* m = &marks[used++];
    m->kind = kind;
    return m;
  }
};
thread_local Profiler t_prof;

// Launch `fn` (returning an sdpa_status) between two profiling events.
template <class F>
int timed(int kind, cudaStream_t s, F&& fn) {
  Profiler::Mark* m = t_prof.next(kind);
  if (m) cudaEventRecord(m->a, s);
  const int rc = fn();
  if (m) cudaEventRecord(m->b, s);
  return rc;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int* error_word() { return static_cast<int*>(device_symbol_address(&g_sdpa_error_word)); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Extent {
  uintptr_t lo, hi;
};
Extent extent(const void* p, size_t bytes) {
  return {reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + bytes};
}
bool overlaps(Extent a, Extent b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

// ---- address-checked build (SDPA_ADDR_CHECK): each entry point registers the
// extents of the buffers it was given; its kernels test every computed access
// against them (addr_ok in common.cuh).
#ifdef SDPA_ADDR_CHECK
constexpr bool kAddrCheck = true;
static __device__ AddrTable g_sdpa_addr_table;
std::atomic<long long> g_addr_shrink{0};

AddrTable* addr_table() { return static_cast<AddrTable*>(device_symbol_address(&g_sdpa_addr_table)); }

// Writes the call's extents (less the debug shrink) ahead of its kernels on
// stream s; the violation counters are left as they are.
AddrTable* bind_extents(std::initializer_list<Extent> ex, int* err, cudaStream_t s) {
  AddrTable* t = addr_table();
  if (!t) return nullptr;
  AddrTable h;
  std::memset(&h, 0, sizeof(h));
  const long long shrink = g_addr_shrink.load(std::memory_order_relaxed);
  for (const Extent& e : ex) {
    if (e.hi <= e.lo || h.n >= (unsigned long long)kAddrExtents) continue;
    const uintptr_t cut = shrink > 0 ? std::min<uintptr_t>((uintptr_t)shrink, e.hi - e.lo) : 0;
    h.lo[h.n] = e.lo;
    h.hi[h.n] = e.hi - cut;
    ++h.n;
  }
  h.err = err;
  // pageable source: the call returns once the bytes are staged, in stream order
  if (cudaMemcpyAsync(t, &h, offsetof(AddrTable, violations), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return nullptr;
  return t;
}
#else
constexpr bool kAddrCheck = false;
AddrTable* bind_extents(std::initializer_list<Extent>, int*, cudaStream_t) { return nullptr; }
#endif

// Rows/heads of the generic row x head x D view (see common.cuh).
void view(const sdpa_problem* p, int& rows_q, int& rows_kv, int& nh_q, int& nh_kv) {
  if (p->layout == SDPA_THD) {
    rows_q = p->total_q;
    rows_kv = p->total_kv;
    nh_q = p->num_heads_q;
    nh_kv = p->num_heads_kv;
  } else if (p->layout == SDPA_BSHD) {
    rows_q = p->batch * p->seqlen_q;
    rows_kv = p->batch * p->seqlen_kv;
    nh_q = p->num_heads_q;
    nh_kv = p->num_heads_kv;
  } else {
    rows_q = p->seqlen_q;
    rows_kv = p->seqlen_kv;
    nh_q = p->batch * p->num_heads_q;
    nh_kv = p->batch * p->num_heads_kv;
  }
}

bool causal(const sdpa_problem* p) { return p->mask_type != SDPA_MASK_NONE; }

// Width of V and O rows (head_dim_v 0 means the symmetric head_dim).
int dv_of(const sdpa_problem* p) { return p->head_dim_v ? p->head_dim_v : p->head_dim; }

// (head_dim, head_dim_v) pairs with a forward kernel: the symmetric 128, 256,
// 512, and (192, 128) (the asymmetric pair the pages' forward engine lists).
bool head_dims_supported(int d, int dv) {
  if (d == dv) return d == 128 || d == 256 || d == 512;
  return d == 192 && dv == 128;
}

int check(const sdpa_problem* p) {
  if (!p) return SDPA_ERR_INVALID_ARG;
  if (p->layout < SDPA_BSHD || p->layout > SDPA_THD) return SDPA_ERR_INVALID_ARG;
  if (p->dtype != SDPA_BF16 && p->dtype != SDPA_FP16) return SDPA_ERR_UNSUPPORTED;
  if (p->mask_type < SDPA_MASK_NONE || p->mask_type > SDPA_MASK_CAUSAL_BOTTOM_RIGHT) return SDPA_ERR_INVALID_ARG;
  if (p->batch < 0 || p->seqlen_q < 0 || p->seqlen_kv < 0) return SDPA_ERR_INVALID_ARG;
  if (p->num_heads_q <= 0 || p->num_heads_kv <= 0) return SDPA_ERR_INVALID_ARG;
  if (p->num_heads_q % p->num_heads_kv) return SDPA_ERR_INVALID_ARG;
  if (p->head_dim_v < 0) return SDPA_ERR_INVALID_ARG;
  if (!head_dims_supported(p->head_dim, dv_of(p))) return SDPA_ERR_UNSUPPORTED;
  if (p->window_left < -1 || p->window_right < -1) return SDPA_ERR_INVALID_ARG;
  if (causal(p) && p->window_right > 0) return SDPA_ERR_INVALID_ARG;
  if (!causal(p) && (p->window_left >= 0 || p->window_right >= 0) && p->seqlen_q != p->seqlen_kv)
    return SDPA_ERR_UNSUPPORTED;
  if (!std::isfinite(p->softmax_scale)) return SDPA_ERR_INVALID_ARG;
  if (p->deterministic != 0 && p->deterministic != 1) return SDPA_ERR_INVALID_ARG;
  if (p->kv_chunk < 0 || p->kv_chunk % 128) return SDPA_ERR_INVALID_ARG;
  if (p->layout == SDPA_THD) {
    if (p->total_q < 0 || p->total_kv < 0) return SDPA_ERR_INVALID_ARG;
  } else if (p->seqlen_q > 0 && p->seqlen_kv == 0 && p->batch > 0) {
    return SDPA_ERR_INVALID_ARG;  // every query would attend an empty key set
  }
  int rq, rk, hq, hk;
  view(p, rq, rk, hq, hk);
  const long long q_elems = (long long)rq * hq * p->head_dim;
  const long long k_elems = (long long)rk * hk * std::max(p->head_dim, dv_of(p));
  if (q_elems >= (1LL << 40) || k_elems >= (1LL << 40)) return SDPA_ERR_UNSUPPORTED;
  if ((long long)p->batch * p->seqlen_q >= (1LL << 31) || (long long)p->batch * p->seqlen_kv >= (1LL << 31))
    return SDPA_ERR_UNSUPPORTED;
  return SDPA_OK;
}

Geom make_geom(const sdpa_problem* p, const int32_t* cu_q, const int32_t* cu_kv) {
  Geom g;
  g.layout = p->layout;
  g.mask = p->mask_type;
  g.batch = p->batch;
  g.sq = p->seqlen_q;
  g.sk = p->seqlen_kv;
  g.hq = p->num_heads_q;
  g.hkv = p->num_heads_kv;
  g.d = p->head_dim;
  g.dv = dv_of(p);
  g.wl = p->window_left;
  g.wr = causal(p) ? 0 : p->window_right;
  g.scale = p->softmax_scale;
  g.scale_log2 = p->softmax_scale * 1.4426950408889634f;
  view(p, g.rows_q, g.rows_kv, g.nh_q, g.nh_kv);
  g.cu_q = cu_q;
  g.cu_kv = cu_kv;
  g.chk = nullptr;
  return g;
}

// 3-D map {D, heads, rows} over a contiguous [rows][heads][D] 16-bit tensor;
// boxes are 64 columns (128 bytes, 128-byte swizzle) x 1 head x box_rows.
int encode(CUtensorMap* m, const void* base, int d, int nh, int rows, int box_rows, bool bf16) {
  auto fn = encode_fn();
  if (!fn) return SDPA_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)nh, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)nh * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SDPA_OK : SDPA_ERR_CUDA;
}

// 3-D map over a contiguous one-byte (E4M3) tensor with 128-byte-swizzled boxes:
// dims[0] is the innermost (contiguous) extent, strides[i] the byte stride of dims[i+1].
int encode_u8(CUtensorMap* m, const void* base, const cuuint64_t (&dims)[3], const cuuint64_t (&strides)[2],
              const cuuint32_t (&box)[3]) {
  auto fn = encode_fn();
  if (!fn) return SDPA_ERR_CUDA;
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SDPA_OK : SDPA_ERR_CUDA;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Keys of the FP8 forward's transposed V per (kv head, d): every sequence's
// keys start on a multiple of 16 (see vt_row0 in fwd_fp8.cu).
size_t fp8_vt_rows(const sdpa_problem* p) {
  if (p->layout == SDPA_THD) return round_up((size_t)p->total_kv + 16 * (size_t)p->batch, 16);
  if (p->layout == SDPA_BSHD) return (size_t)p->batch * round_up((size_t)p->seqlen_kv, 16);
  return round_up((size_t)p->seqlen_kv, 16);
}

// FP8 forward: head_dim 128 or 256, equal for Q/K and V (PR #3527 "Scope"
// serves FP8 at head dims up to 256).
int check_fp8(const sdpa_problem* p) {
  const int rc = check(p);
  if (rc) return rc;
  return ((p->head_dim == 128 || p->head_dim == 256) && dv_of(p) == p->head_dim) ? SDPA_OK : SDPA_ERR_UNSUPPORTED;
}

// Key tiles one 128-row query tile can touch (the slot count of the head_dim
// 256/512 tile arrays): the whole key range, or the window's span.
int kv_slots(const sdpa_problem* p) {
  const int nkt = (p->seqlen_kv + 127) / 128;
  const int wr = causal(p) ? 0 : p->window_right;
  if (p->window_left >= 0 && wr >= 0) {
    const long long span = 128LL + p->window_left + wr;  // keys one query tile can see
    return (int)std::min<long long>(nkt, span / 128 + 2);
  }
  return nkt;
}

// Key-tile chunking of the head_dim 256/512 backward (bwd_big.cu): the P / dS
// tile arrays hold one chunk of key tiles at a time, so their size does not
// grow with the key length (TransformerEngine PR #3527, "Known limitations":
// the prior art's workspace grows to 74 GiB at 64k tokens and caps the
// context). A bounded (left, right) window already bounds the key tiles one
// query tile sees; otherwise the chunk is as many key tiles as fit the
// budget below (at least one).
constexpr size_t kBwdTileBudget = size_t(512) << 20;

struct BigPlan {
  int chunk;   // key tiles per chunk
  int slots;   // tile slots per (batch, q head, q tile)
  int chunks;  // number of chunks
};
BigPlan big_plan(const sdpa_problem* p) {
  const int nkt = (p->seqlen_kv + 127) / 128;
  const int kvs = kv_slots(p);
  const size_t tile_bytes = 2 * 32768;  // the P and dS images of one (query tile, key tile) pair
  const size_t per_slot = (size_t)p->batch * p->num_heads_q * ((p->seqlen_q + 127) / 128) * tile_bytes;
  const int wr = causal(p) ? 0 : p->window_right;
  BigPlan pl;
  if (p->kv_chunk > 0) {  // the caller's chunk
    pl.chunk = std::max(1, std::min(nkt, p->kv_chunk / 128));
    pl.slots = std::min(pl.chunk, kvs);
  } else if ((p->window_left >= 0 && wr >= 0) || (size_t)kvs * per_slot <= kBwdTileBudget || nkt <= 1) {
    pl.chunk = std::max(nkt, 1);
    pl.slots = kvs;
  } else {
    pl.chunk = (int)std::max<size_t>(1, std::min<size_t>(kBwdTileBudget / std::max<size_t>(per_slot, 1), nkt));
    pl.slots = std::min(pl.chunk, kvs);
  }
  pl.chunks = (nkt + pl.chunk - 1) / pl.chunk;
  return pl;
}

// Backward workspace carve-up. head_dim 128: per-row statistics and the fp32
// dQ accumulator. head_dim 256/512: statistics, the fp32 dQ accumulator when
// the key tiles are split into chunks, and the 16-bit P / dS tile arrays of
// one chunk.
struct BwdWs {
  size_t guard_off, order_off, lse2_off, delta_off, acc_off, ptile_off, dstile_off, total;
  int stat_rows;
  bool has_acc;
};
BwdWs bwd_ws(const sdpa_problem* p) {
  int rq, rk, hq, hk;
  view(p, rq, rk, hq, hk);
  BwdWs w;
  // rows of the per-head statistics arrays (see SeqInfo::srow0), plus 128 rows of
  // padding for query tiles that overhang the last sequence
  size_t srows;
  if (p->layout == SDPA_THD)
    srows = round_up((size_t)p->total_q + 4 * (size_t)p->batch + 3, 4);
  else if (p->layout == SDPA_BSHD)
    srows = (size_t)p->batch * round_up((size_t)p->seqlen_q, 4);
  else
    srows = round_up((size_t)p->seqlen_q, 4);
  w.stat_rows = (int)(srows + 128);
  w.guard_off = 0;
  // THD, head_dim 128: the sequence order the guard writes (longest first)
  const bool ordered = p->layout == SDPA_THD && p->head_dim == 128;
  w.order_off = ordered ? 256 : 0;
  w.lse2_off = ordered ? 256 + round_up((size_t)p->batch * 4, 256) : 256;
  w.delta_off = round_up(w.lse2_off + (size_t)hq * w.stat_rows * 4, 256);
  const size_t after_stats = round_up(w.delta_off + (size_t)hq * w.stat_rows * 4, 256);
  const size_t acc_bytes = (size_t)hq * rq * p->head_dim * 4;
  if (p->head_dim == 128) {
    // the deterministic backward writes dQ directly and needs no accumulator
    w.acc_off = after_stats;
    w.has_acc = !p->deterministic;
    w.ptile_off = w.dstile_off = 0;
    w.total = p->deterministic ? after_stats : round_up(w.acc_off + acc_bytes, 256);
  } else {
    const BigPlan pl = big_plan(p);
    const size_t tiles = (size_t)p->batch * p->num_heads_q * ((p->seqlen_q + 127) / 128) * pl.slots;
    w.has_acc = pl.chunks > 1;
    w.acc_off = after_stats;
    const size_t after_acc = w.has_acc ? w.acc_off + acc_bytes : after_stats;
    w.ptile_off = round_up(after_acc, 1024);
    w.dstile_off = w.ptile_off + tiles * 32768;
    w.total = w.dstile_off + tiles * 32768;
  }
  return w;
}

// kv heads whose key tiles interleave in the D128 backward grid: the largest
// divisor of num_heads_kv whose query-side rows (Q and dO, plus the fp32 dQ
// accumulator unless deterministic) fit in 128 MiB, about the L2. Interleaving
// heads lets the heavy first key tiles of every head start early; keeping their
// rows within the L2 keeps the CTAs that walk the same rows from re-reading
// them from HBM.
int bwd_head_block(const sdpa_problem* p) {
  const int group = p->num_heads_q / p->num_heads_kv;
  const size_t per_head = (size_t)p->seqlen_q * group * p->head_dim * (p->deterministic ? 4 : 8);
  int hb = 1;
  for (int d = 1; d <= p->num_heads_kv; ++d)
    if (p->num_heads_kv % d == 0 && (size_t)d * per_head <= (size_t)128 << 20) hb = d;
  return hb;
}

}  // namespace

static std::atomic<int> g_max_ctas{0};
int debug_max_ctas() { return g_max_ctas.load(std::memory_order_relaxed); }

// Unique ID of the calling thread's current context (cuCtxGetId; IDs are not
// reused within a process), 0 when there is none or the driver lacks the call.
static unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(ptr);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

void* device_symbol_address(const void* symbol) {
  struct Entry {
    const void* symbol;
    int dev;
    unsigned long long ctx;
    void* addr;
  };
  static std::mutex mu;
  static Entry cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  Entry* slot = nullptr;
  for (Entry& e : cache) {
    if (e.symbol == symbol && e.dev == dev) {
      slot = &e;
      break;
    }
    if (!slot && !e.symbol) slot = &e;  // first free entry, unless a match follows
  }
  if (slot && slot->symbol == symbol && slot->dev == dev && ctx != 0 && slot->ctx == ctx) return slot->addr;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, symbol) != cudaSuccess || !addr) return nullptr;
  const unsigned long long now = current_context_id();  // the lookup may have made the context current
  if (slot && now != 0) *slot = Entry{symbol, dev, now, addr};
  return addr;
}

int set_kernel_smem(const void* kernel, int bytes, int carveout) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;  // (kernel, device) already configured
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return SDPA_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return SDPA_ERR_CUDA;
  if (carveout >= 0 && cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout) !=
                           cudaSuccess)
    return SDPA_ERR_CUDA;
  done.insert({kernel, dev});
  return SDPA_OK;
}

}  // namespace sdpa

using namespace sdpa;

extern "C" {

int sdpa_check_problem(const sdpa_problem* p) { return check(p); }

size_t sdpa_fwd_workspace_size(const sdpa_problem* p) {
  if (check(p) != SDPA_OK) return 0;
  // THD: the metadata guard word at offset 0; head_dim 128: the tile ticket
  // counter of the persistent kernel at offset 128
  return (p->layout == SDPA_THD || p->head_dim == 128) ? 256 : 0;
}

size_t sdpa_bwd_workspace_size(const sdpa_problem* p) {
  if (check(p) != SDPA_OK || dv_of(p) != p->head_dim) return 0;
  return bwd_ws(p).total;
}

int sdpa_fwd(const sdpa_problem* p, const void* q, const void* k, const void* v, void* o, float* lse,
             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, void* workspace, size_t ws_bytes,
             void* stream) {
  t_last_launches = 0;
  int rc = check(p);
  if (rc) return rc;
  int rq, rk, hq, hk;
  view(p, rq, rk, hq, hk);
  const bool thd = p->layout == SDPA_THD;
  if (p->batch == 0 || rq == 0) return SDPA_OK;
  if (!q || !k || !v || !o || !lse) return SDPA_ERR_INVALID_ARG;
  if (thd && (!cu_seqlens_q || !cu_seqlens_kv)) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return SDPA_ERR_ALIGNMENT;
  const size_t need = sdpa_fwd_workspace_size(p);
  if (ws_bytes < need || (need && !workspace)) return SDPA_ERR_WORKSPACE_TOO_SMALL;
  if (need && !aligned16(workspace)) return SDPA_ERR_ALIGNMENT;
  const size_t qb = (size_t)rq * hq * p->head_dim * 2, kb = (size_t)rk * hk * p->head_dim * 2;
  const size_t vb = (size_t)rk * hk * dv_of(p) * 2, ob = (size_t)rq * hq * dv_of(p) * 2;
  const Extent eo = extent(o, ob), el = extent(lse, (size_t)rq * hq * 4);
  for (Extent in : {extent(q, qb), extent(k, kb), extent(v, vb)})
    if (overlaps(eo, in) || overlaps(el, in)) return SDPA_ERR_OVERLAP;
  if (overlaps(eo, el)) return SDPA_ERR_OVERLAP;
  if (need && (overlaps(extent(workspace, need), eo) || overlaps(extent(workspace, need), el)))
    return SDPA_ERR_OVERLAP;

  int* err = error_word();
  if (!err) return SDPA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = p->dtype == SDPA_BF16;
  FwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  L.p.g = make_geom(p, cu_seqlens_q, cu_seqlens_kv);
  const size_t cub = thd ? 4 * ((size_t)p->batch + 1) : 0;
  L.p.g.chk = bind_extents({extent(q, qb), extent(k, kb), extent(v, vb), eo, el, extent(cu_seqlens_q, cub),
                            extent(cu_seqlens_kv, cub), extent(workspace, need)},
                           err, s);
  if (kAddrCheck && !L.p.g.chk) return SDPA_ERR_CUDA;
  L.p.o = o;
  L.p.lse = lse;
  L.p.err = err;
  L.p.guard = thd ? static_cast<const int*>(workspace) : nullptr;
  L.p.n_q_tiles = (p->seqlen_q + 127) / 128;
  L.p.dv_splits = p->head_dim == 512 ? 2 : 1;
  L.p.tile_counter = p->head_dim == 128 ? reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + 128) : nullptr;
  L.stream = s;
  const int dv_cta = dv_of(p) == 512 ? 256 : dv_of(p);  // value columns one CTA accumulates
  if ((rc = encode(&L.tmQ, q, p->head_dim, hq, rq, 128, bf16))) return rc;
  if ((rc = encode(&L.tmK, k, p->head_dim, hk, rk, 128, bf16))) return rc;
  if ((rc = encode(&L.tmV, v, dv_of(p), hk, rk, 32768 / (dv_cta * 2), bf16))) return rc;
  int launches = 0;
  if (thd) {
    rc = timed(SDPA_KERNEL_GUARD, s,
               [&] { return launch_guard(L.p.g, p->total_q, p->total_kv, static_cast<int*>(workspace), err, s); });
    if (rc) return rc;
    ++launches;
  }
  if ((rc = timed(SDPA_KERNEL_FWD, s, [&] { return launch_fwd(L, p->head_dim, dv_of(p), bf16); }))) return rc;
  ++launches;
  t_last_launches = launches;
  return SDPA_OK;
}

int sdpa_bwd(const sdpa_problem* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
             const int32_t* cu_seqlens_kv, void* workspace, size_t ws_bytes, void* stream) {
  t_last_launches = 0;
  int rc = check(p);
  if (rc) return rc;
  if (dv_of(p) != p->head_dim) return SDPA_ERR_UNSUPPORTED;  // the backward is symmetric only
  int rq, rk, hq, hk;
  view(p, rq, rk, hq, hk);
  const bool thd = p->layout == SDPA_THD;
  if (p->batch == 0 || (rq == 0 && rk == 0)) return SDPA_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return SDPA_ERR_INVALID_ARG;
  if (thd && (!cu_seqlens_q || !cu_seqlens_kv)) return SDPA_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, o, (const void*)lse, dout, (const void*)dq, (const void*)dk, (const void*)dv})
    if (!aligned16(ptr)) return SDPA_ERR_ALIGNMENT;
  const BwdWs w = bwd_ws(p);
  if (ws_bytes < w.total || !workspace) return SDPA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SDPA_ERR_ALIGNMENT;
  const size_t qb = (size_t)rq * hq * p->head_dim * 2, kb = (size_t)rk * hk * p->head_dim * 2;
  const Extent outs[4] = {extent(dq, qb), extent(dk, kb), extent(dv, kb), extent(workspace, w.total)};
  const Extent ins[6] = {extent(q, qb), extent(k, kb), extent(v, kb), extent(o, qb), extent(lse, (size_t)rq * hq * 4),
                         extent(dout, qb)};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], ins[b])) return SDPA_ERR_OVERLAP;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], outs[b])) return SDPA_ERR_OVERLAP;
  }

  int* err = error_word();
  if (!err) return SDPA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = p->dtype == SDPA_BF16;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* guard = thd ? reinterpret_cast<int*>(ws + w.guard_off) : nullptr;
  int* order = w.order_off ? reinterpret_cast<int*>(ws + w.order_off) : nullptr;
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2_off);
  float* delta = reinterpret_cast<float*>(ws + w.delta_off);
  float* acc = reinterpret_cast<float*>(ws + w.acc_off);
  Geom g = make_geom(p, cu_seqlens_q, cu_seqlens_kv);
  const size_t cub = thd ? 4 * ((size_t)p->batch + 1) : 0;
  g.chk = bind_extents({outs[0], outs[1], outs[2], outs[3], ins[0], ins[1], ins[2], ins[3], ins[4], ins[5],
                        extent(cu_seqlens_q, cub), extent(cu_seqlens_kv, cub)},
                       err, s);
  if (kAddrCheck && !g.chk) return SDPA_ERR_CUDA;
  int launches = 0;
  if (thd) {
    if ((rc = timed(SDPA_KERNEL_GUARD, s, [&] { return launch_guard(g, p->total_q, p->total_kv, guard, err, s, order); })))
      return rc;
    ++launches;
  }
  PrepParams pp;
  pp.g = g;
  pp.o = o;
  pp.dout = dout;
  pp.lse = lse;
  pp.lse2 = lse2;
  pp.delta = delta;
  pp.stat_rows = w.stat_rows;
  pp.dq_acc = w.has_acc ? acc : nullptr;
  pp.guard = guard;
  if ((rc = timed(SDPA_KERNEL_PREPROCESS, s, [&] { return launch_preprocess(pp, bf16, s); }))) return rc;
  ++launches;

  if (p->head_dim != 128) {
    BigBwdLaunch B;
    std::memset(&B, 0, sizeof(B));
    B.p.g = g;
    B.p.p_tiles = ws + w.ptile_off;
    B.p.ds_tiles = ws + w.dstile_off;
    B.p.nlse2 = lse2;
    B.p.delta = delta;
    B.p.stat_rows = w.stat_rows;
    B.p.dq = dq;
    B.p.dk = dk;
    B.p.dv = dv;
    B.p.err = err;
    B.p.guard = guard;
    B.p.n_q_tiles = (p->seqlen_q + 127) / 128;
    B.p.n_kv_tiles = (p->seqlen_kv + 127) / 128;
    const BigPlan pl = big_plan(p);
    B.p.slots = pl.slots;
    B.p.chunk = pl.chunk;
    B.p.chunk_lo = 0;
    B.p.chunk_hi = B.p.n_kv_tiles;
    B.p.dq_acc = w.has_acc ? acc : nullptr;
    B.stream = s;
    if ((rc = encode(&B.tmQ, q, p->head_dim, hq, rq, 128, bf16))) return rc;
    if ((rc = encode(&B.tmDO, dout, p->head_dim, hq, rq, 128, bf16))) return rc;
    if ((rc = encode(&B.tmK, k, p->head_dim, hk, rk, 128, bf16))) return rc;
    if ((rc = encode(&B.tmV, v, p->head_dim, hk, rk, 128, bf16))) return rc;
    if ((rc = encode(&B.tmQ64, q, p->head_dim, hq, rq, 64, bf16))) return rc;
    if ((rc = encode(&B.tmDO64, dout, p->head_dim, hq, rq, 64, bf16))) return rc;
    if ((rc = encode(&B.tmK64, k, p->head_dim, hk, rk, 64, bf16))) return rc;
    int n = 0;
    if ((rc = timed(SDPA_KERNEL_BWD, s, [&] { return launch_bwd_big(B, p->head_dim, bf16, &n); }))) return rc;
    launches += n;
    if (w.has_acc) {  // dQ summed over the key-tile chunks: scale and convert once
      if ((rc = timed(SDPA_KERNEL_DQ_FINALIZE, s, [&] { return launch_dq_finalize(g, acc, dq, guard, bf16, s); })))
        return rc;
      ++launches;
    }
    t_last_launches = launches;
    return SDPA_OK;
  }

  BwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  L.p.g = g;
  L.p.dq_acc = acc;
  L.p.lse2 = lse2;
  L.p.delta = delta;
  L.p.stat_rows = w.stat_rows;
  L.p.dk = dk;
  L.p.dv = dv;
  L.p.err = err;
  L.p.guard = guard;
  L.p.order = order;
  L.p.head_block = bwd_head_block(p);
  L.p.n_kv_tiles = (p->seqlen_kv + 127) / 128;
  L.stream = s;
  if ((rc = encode(&L.tmQ, q, p->head_dim, hq, rq, 64, bf16))) return rc;
  if ((rc = encode(&L.tmDO, dout, p->head_dim, hq, rq, 64, bf16))) return rc;
  if ((rc = encode(&L.tmK, k, p->head_dim, hk, rk, 128, bf16))) return rc;
  if ((rc = encode(&L.tmV, v, p->head_dim, hk, rk, 128, bf16))) return rc;
  const bool det = p->deterministic != 0;
  L.p.dq_acc = det ? nullptr : acc;
  int n = 0;
  if ((rc = timed(SDPA_KERNEL_BWD, s, [&] { return launch_bwd_dkdv(L, p->head_dim, bf16, !det, &n); }))) return rc;
  launches += n;
  if (det) {
    // dQ per query tile, key tiles in a fixed order, written once
    DqLaunch Dq;
    std::memset(&Dq, 0, sizeof(Dq));
    Dq.p.g = g;
    Dq.p.dq = dq;
    Dq.p.nlse2 = lse2;
    Dq.p.delta = delta;
    Dq.p.stat_rows = w.stat_rows;
    Dq.p.err = err;
    Dq.p.guard = guard;
    Dq.p.n_q_tiles = (p->seqlen_q + 127) / 128;
    Dq.stream = s;
    if ((rc = encode(&Dq.tmQ, q, p->head_dim, hq, rq, 128, bf16))) return rc;
    if ((rc = encode(&Dq.tmDO, dout, p->head_dim, hq, rq, 128, bf16))) return rc;
    if ((rc = encode(&Dq.tmK, k, p->head_dim, hk, rk, 128, bf16))) return rc;
    if ((rc = encode(&Dq.tmV, v, p->head_dim, hk, rk, 128, bf16))) return rc;
    if ((rc = timed(SDPA_KERNEL_BWD_DQ, s, [&] { return launch_dq128(Dq, bf16); }))) return rc;
    ++launches;
  } else {
    if ((rc = timed(SDPA_KERNEL_DQ_FINALIZE, s, [&] { return launch_dq_finalize(g, acc, dq, guard, bf16, s); })))
      return rc;
    ++launches;
  }
  t_last_launches = launches;
  return SDPA_OK;
}

size_t sdpa_fwd_fp8_workspace_size(const sdpa_problem* p) {
  if (check_fp8(p) != SDPA_OK) return 0;
  int rq, rk, hq, hk;
  view(p, rq, rk, hq, hk);
  return 256 + (size_t)hk * p->head_dim * fp8_vt_rows(p);
}

int sdpa_fwd_fp8(const sdpa_problem* p, const void* q8, const void* k8, const void* v8, float descale_q,
                 float descale_k, float descale_v, void* o, float* lse, const int32_t* cu_seqlens_q,
                 const int32_t* cu_seqlens_kv, void* workspace, size_t ws_bytes, void* stream) {
  t_last_launches = 0;
  int rc = check_fp8(p);
  if (rc) return rc;
  if (!std::isfinite(descale_q) || !std::isfinite(descale_k) || !std::isfinite(descale_v) || !(descale_q > 0.f) ||
      !(descale_k > 0.f) || !(descale_v > 0.f))
    return SDPA_ERR_INVALID_ARG;
  int rq, rk, hq, hk;
  view(p, rq, rk, hq, hk);
  const bool thd = p->layout == SDPA_THD;
  if (p->batch == 0 || rq == 0) return SDPA_OK;
  if (!q8 || !k8 || !v8 || !o || !lse) return SDPA_ERR_INVALID_ARG;
  if (thd && (!cu_seqlens_q || !cu_seqlens_kv)) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned16(lse))
    return SDPA_ERR_ALIGNMENT;
  const size_t need = sdpa_fwd_fp8_workspace_size(p);
  if (ws_bytes < need || !workspace) return SDPA_ERR_WORKSPACE_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SDPA_ERR_ALIGNMENT;
  const size_t D = (size_t)p->head_dim;
  const size_t qb = (size_t)rq * hq * D, kb = (size_t)rk * hk * D, ob = (size_t)rq * hq * D * 2;
  const Extent outs[3] = {extent(o, ob), extent(lse, (size_t)rq * hq * 4), extent(workspace, need)};
  const Extent ins[3] = {extent(q8, qb), extent(k8, kb), extent(v8, kb)};
  for (int x = 0; x < 3; ++x) {
    for (int y = 0; y < 3; ++y)
      if (overlaps(outs[x], ins[y])) return SDPA_ERR_OVERLAP;
    for (int y = x + 1; y < 3; ++y)
      if (overlaps(outs[x], outs[y])) return SDPA_ERR_OVERLAP;
  }
  int* err = error_word();
  if (!err) return SDPA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Fp8Launch L;
  std::memset(&L, 0, sizeof(L));
  L.p.g = make_geom(p, cu_seqlens_q, cu_seqlens_kv);
  const size_t cub = thd ? 4 * ((size_t)p->batch + 1) : 0;
  L.p.g.chk = bind_extents({outs[0], outs[1], outs[2], ins[0], ins[1], ins[2], extent(cu_seqlens_q, cub),
                            extent(cu_seqlens_kv, cub)},
                           err, s);
  if (kAddrCheck && !L.p.g.chk) return SDPA_ERR_CUDA;
  L.p.g.scale = p->softmax_scale * descale_q * descale_k;  // scores of the decoded codes
  L.p.g.scale_log2 = L.p.g.scale * 1.4426950408889634f;
  L.p.v = static_cast<const uint8_t*>(v8);
  L.p.vt = ws + 256;
  L.p.tile_counter = reinterpret_cast<int*>(ws + 128);
  L.p.vt_rows = (int)fp8_vt_rows(p);
  L.p.o = o;
  L.p.lse = lse;
  L.p.err = err;
  L.p.guard = thd ? reinterpret_cast<const int*>(ws) : nullptr;
  L.p.n_q_tiles = (p->seqlen_q + 127) / 128;
  L.p.o_scale = descale_v / 448.f;
  L.stream = s;
  if ((size_t)L.p.vt_rows * hk * D >= (1ull << 40)) return SDPA_ERR_UNSUPPORTED;
  {
    // Q, K: boxes of 128 one-byte columns (a head_dim 256 tile is two); Vt: one box of D rows
    const cuuint64_t dq[3] = {D, (cuuint64_t)hq, (cuuint64_t)(rq > 0 ? rq : 1)};
    const cuuint64_t sq[2] = {D, (cuuint64_t)hq * D};
    const cuuint64_t dk[3] = {D, (cuuint64_t)hk, (cuuint64_t)(rk > 0 ? rk : 1)};
    const cuuint64_t sk[2] = {D, (cuuint64_t)hk * D};
    const cuuint64_t dvt[3] = {(cuuint64_t)L.p.vt_rows, D, (cuuint64_t)hk};
    const cuuint64_t svt[2] = {(cuuint64_t)L.p.vt_rows, (cuuint64_t)L.p.vt_rows * D};
    const cuuint32_t box_rows[3] = {128, 1, 128}, box_vt[3] = {128, (cuuint32_t)D, 1};
    if ((rc = encode_u8(&L.tmQ, q8, dq, sq, box_rows))) return rc;
    if ((rc = encode_u8(&L.tmK, k8, dk, sk, box_rows))) return rc;
    if ((rc = encode_u8(&L.tmVt, L.p.vt, dvt, svt, box_vt))) return rc;
  }
  int launches = 0;
  if (thd) {
    if ((rc = timed(SDPA_KERNEL_GUARD, s,
                    [&] { return launch_guard(L.p.g, p->total_q, p->total_kv, reinterpret_cast<int*>(ws), err, s); })))
      return rc;
    ++launches;
  }
  if ((rc = timed(SDPA_KERNEL_V_TRANSPOSE, s, [&] { return launch_vt(L.p, s); }))) return rc;
  ++launches;
  if ((rc = timed(SDPA_KERNEL_FWD, s, [&] { return launch_fwd_fp8(L, p->dtype == SDPA_BF16); }))) return rc;
  ++launches;
  t_last_launches = launches;
  return SDPA_OK;
}

int sdpa_merge(const sdpa_merge_problem* p, const void* o_parts, const float* lse_parts, void* o, float* lse,
               void* stream) {
  t_last_launches = 0;
  if (!p) return SDPA_ERR_INVALID_ARG;
  if (p->n_parts < 1 || p->n_parts > 64 || p->items < 0) return SDPA_ERR_INVALID_ARG;
  if (p->dtype != SDPA_BF16 && p->dtype != SDPA_FP16) return SDPA_ERR_UNSUPPORTED;
  if (p->head_dim != 128 && p->head_dim != 256 && p->head_dim != 512) return SDPA_ERR_UNSUPPORTED;
  if (p->items == 0) return SDPA_OK;
  if (!o_parts || !lse_parts || !o || !lse) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o) || !aligned16(lse)) return SDPA_ERR_ALIGNMENT;
  const size_t ob = (size_t)p->items * p->head_dim * 2, lb = (size_t)p->items * 4;
  const Extent eo = extent(o, ob), el = extent(lse, lb);
  for (Extent in : {extent(o_parts, ob * p->n_parts), extent(lse_parts, lb * p->n_parts)})
    if (overlaps(eo, in) || overlaps(el, in)) return SDPA_ERR_OVERLAP;
  if (overlaps(eo, el)) return SDPA_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AddrTable* chk = bind_extents({eo, el, extent(o_parts, ob * p->n_parts), extent(lse_parts, lb * p->n_parts)},
                                error_word(), s);
  if (kAddrCheck && !chk) return SDPA_ERR_CUDA;
  const int rc = timed(SDPA_KERNEL_MERGE, s, [&] {
    return launch_merge(o_parts, lse_parts, o, lse, p->items, p->head_dim, p->n_parts, p->dtype == SDPA_BF16, chk,
                        s);
  });
  if (rc) return rc;
  t_last_launches = 1;
  return SDPA_OK;
}

int sdpa_get_device_error(void* stream) {
  int* err = error_word();
  if (!err) return SDPA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SDPA_ERR_CUDA;
  int host = 0;
  if (cudaMemcpyFromSymbol(&host, g_sdpa_error_word, sizeof(int)) != cudaSuccess) return SDPA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_sdpa_error_word, &zero, sizeof(int)) != cudaSuccess) return SDPA_ERR_CUDA;
  return host;
}

const char* sdpa_error_string(int status) {
  switch (status) {
    case SDPA_OK: return "ok";
    case SDPA_ERR_INVALID_ARG: return "invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "unsupported problem (dtype, head_dim, layout or mask/window combination)";
    case SDPA_ERR_ALIGNMENT: return "a device pointer is not 16-byte aligned";
    case SDPA_ERR_OVERLAP: return "an output buffer overlaps another buffer";
    case SDPA_ERR_WORKSPACE_TOO_SMALL: return "workspace missing or smaller than the required size";
    case SDPA_ERR_BAD_SEQLENS: return "cu_seqlens rejected by the device-side guard";
    case SDPA_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    case SDPA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case SDPA_ERR_ADDRESS: return "a kernel access fell outside the call's buffers (address-checked library)";
    default: return "unknown status";
  }
}

int sdpa_last_launch_count(void) { return t_last_launches; }

int sdpa_debug_set_max_ctas(int max_ctas) {
  if (max_ctas < 0) return SDPA_ERR_INVALID_ARG;
  g_max_ctas.store(max_ctas, std::memory_order_relaxed);
  return SDPA_OK;
}

int sdpa_debug_address_report(unsigned long long* violations, unsigned long long* first_addr,
                              unsigned long long* first_bytes) {
#ifdef SDPA_ADDR_CHECK
  AddrTable* t = addr_table();
  if (!t || cudaDeviceSynchronize() != cudaSuccess) return SDPA_ERR_CUDA;
  unsigned long long v[3] = {0, 0, 0};
  uint8_t* counters = reinterpret_cast<uint8_t*>(t) + offsetof(AddrTable, violations);
  if (cudaMemcpy(v, counters, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SDPA_ERR_CUDA;
  const unsigned long long zero[3] = {0, 0, 0};
  if (cudaMemcpy(counters, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SDPA_ERR_CUDA;
  if (violations) *violations = v[0];
  if (first_addr) *first_addr = v[1];
  if (first_bytes) *first_bytes = v[2];
  return SDPA_OK;
#else
  (void)violations;
  (void)first_addr;
  (void)first_bytes;
  return SDPA_ERR_UNSUPPORTED;
#endif
}

int sdpa_debug_address_shrink(long long bytes) {
#ifdef SDPA_ADDR_CHECK
  if (bytes < 0) return SDPA_ERR_INVALID_ARG;
  g_addr_shrink.store(bytes, std::memory_order_relaxed);
  return SDPA_OK;
#else
  (void)bytes;
  return SDPA_ERR_UNSUPPORTED;
#endif
}

int sdpa_selftest_bounded_wait(unsigned limit_us, void* stream) {
  int* err = error_word();
  if (!err) return SDPA_ERR_CUDA;
  if (limit_us == 0 || limit_us > 1000000u) return SDPA_ERR_INVALID_ARG;
  return launch_wait_selftest((uint64_t)limit_us * 1000ull, err, static_cast<cudaStream_t>(stream));
}

int sdpa_profile_begin(void) {
  t_prof.on = true;
  t_prof.used = 0;
  return SDPA_OK;
}

int sdpa_profile_end(double* ms_by_kind, int* launches_by_kind, int n_kinds) {
  if (n_kinds < 0 || (n_kinds > 0 && (!ms_by_kind || !launches_by_kind))) return SDPA_ERR_INVALID_ARG;
  for (int k = 0; k < n_kinds; ++k) {
    ms_by_kind[k] = 0.0;
    launches_by_kind[k] = 0;
  }
  int rc = SDPA_OK;
  for (size_t i = 0; i < t_prof.used; ++i) {
    const Profiler::Mark& m = t_prof.marks[i];
    float ms = 0.f;
    if (cudaEventSynchronize(m.b) != cudaSuccess || cudaEventElapsedTime(&ms, m.a, m.b) != cudaSuccess) {
      rc = SDPA_ERR_CUDA;
      continue;
    }
    if (m.kind < n_kinds) {
      ms_by_kind[m.kind] += ms;
      launches_by_kind[m.kind] += 1;
    }
  }
  t_prof.on = false;
  t_prof.used = 0;
  return rc;
}

}  // extern "C"
