// aux.cu -- the memory-bound steps around the attention kernels:
//   * the THD metadata guard (TransformerEngine PR #3705, "Execution and
//     supported scope": compactness is checked on the GPU on every
//     execution -- zero-based cumulative lengths, valid bounds, non-empty KV
//     for live Q);
//   * the backward preprocess: delta = rowsum(dO * O) in fp32, -LSE*log2(e)
//     (-inf for rows without keys), and the fp32 dQ accumulator zeroed;
//   * the dQ finalise: dQ = scale * accumulator, cast to the input dtype.
#include <algorithm>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

// order (may be null): the sequence indices ordered by query-tile count,
// longest first -- a counting sort over min(max_q/64 + 1, kOrderBins) bins,
// so it is a permutation of [0, batch) whatever the lengths hold. Sequences
// of one bin keep no fixed order among themselves; the order only decides
// when a sequence's CTAs start, never what they compute.
constexpr int kOrderBins = 4096;

__device__ __forceinline__ int order_bin(int lq, int n_bins) {
  if (lq <= 0) return 0;
  const int t = (lq - 1) / 64 + 1;
  return t < n_bins ? t : n_bins - 1;
}

__global__ void __launch_bounds__(256) guard_kernel(const int32_t* cu_q, const int32_t* cu_kv, int batch, int total_q,
                                                    int total_kv, int max_q, int max_kv, int* guard, int* err,
                                                    int* order, int n_bins, AddrTable* chk) {
  __shared__ int bad;
  __shared__ int bins[kOrderBins];
  __shared__ int warp_sum[8];
  // the address-checked build reads the two arrays and writes the guard word
  // and the order only where the call registered them (else: rejected)
  const bool in_bounds = SDPA_ADDR_OK(chk, cu_q, 4ull * (batch + 1)) && SDPA_ADDR_OK(chk, cu_kv, 4ull * (batch + 1)) &&
                         SDPA_ADDR_OK(chk, guard, 4) && (!order || SDPA_ADDR_OK(chk, order, 4ull * batch));
  if (!in_bounds) {
    if (threadIdx.x == 0 && SDPA_ADDR_OK(chk, guard, 4)) *guard = SDPA_ERR_ADDRESS;
    return;
  }
  if (threadIdx.x == 0) bad = (cu_q[0] != 0) || (cu_kv[0] != 0) || (cu_q[batch] != total_q) || (cu_kv[batch] != total_kv);
  if (order)
    for (int x = threadIdx.x; x < n_bins; x += blockDim.x) bins[x] = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    const int lq = cu_q[b + 1] - cu_q[b];
    const int lk = cu_kv[b + 1] - cu_kv[b];
    if (lq < 0 || lk < 0 || lq > max_q || lk > max_kv || (lq > 0 && lk == 0)) atomicOr(&bad, 1);
    if (order) atomicAdd(&bins[order_bin(lq, n_bins)], 1);
  }
  __syncthreads();
  if (order) {
    // bins[x] <- sequences in bins above x (exclusive scan from the top):
    // thread t owns the bins n_bins-1-per*t ... n_bins-per*(t+1)
    const int per = (n_bins + blockDim.x - 1) / blockDim.x;
    int own = 0;
    for (int j = 0; j < per; ++j) {
      const int x = n_bins - 1 - (per * (int)threadIdx.x + j);
      if (x >= 0) own += bins[x];
    }
    const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
    int incl = own;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    int run = incl - own;
    for (int w = 0; w < wid; ++w) run += warp_sum[w];
    for (int j = 0; j < per; ++j) {
      const int x = n_bins - 1 - (per * (int)threadIdx.x + j);
      if (x >= 0) {
        const int c = bins[x];
        bins[x] = run;
        run += c;
      }
    }
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += blockDim.x)
      order[atomicAdd(&bins[order_bin(cu_q[b + 1] - cu_q[b], n_bins)], 1)] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *guard = bad ? SDPA_ERR_BAD_SEQLENS : 0;
    if (bad) record_error(err, SDPA_ERR_BAD_SEQLENS);
  }
}

int launch_guard(const Geom& g, int total_q, int total_kv, int* guard, int* err, cudaStream_t s, int* order) {
  const int n_bins = std::min(g.sq / 64 + 2, kOrderBins);
  guard_kernel<<<1, 256, 0, s>>>(g.cu_q, g.cu_kv, g.batch, total_q, total_kv, g.sq, g.sk, guard, err, order, n_bins,
                                 g.chk);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

// Statistics row of generic query row `row` (its query position in its
// sequence, plus the sequence's block start SeqInfo::srow0): BSHD and SBHD by
// arithmetic, THD by a binary search of cu_seqlens_q (rows are tokens).
__device__ __forceinline__ int stat_row(const Geom& g, int row) {
  if (g.layout == SDPA_SBHD) return row;
  if (g.layout == SDPA_BSHD) {
    const int b = row / g.sq;
    return b * ((g.sq + 3) & ~3) + (row - b * g.sq);
  }
  int lo = 0, hi = g.batch;  // the b with cu_q[b] <= row < cu_q[b + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (SDPA_ADDR_OK(g.chk, g.cu_q + mid, 4) && g.cu_q[mid] <= row)
      lo = mid;
    else
      hi = mid;
  }
  const int c0 = SDPA_ADDR_OK(g.chk, g.cu_q + lo, 4) ? g.cu_q[lo] : 0;
  return ((c0 + 3) & ~3) + 4 * lo + (row - c0);
}

// delta = rowsum(dO * O) and -LSE*log2(e) for every (query row, head) item of
// the generic view. The items of O, dO and the token-major LSE are contiguous
// in every layout (item = row * nh_q + head), so the whole grid strides over
// them evenly whatever the sequence lengths; G lanes share an item, each lane
// holding two 16-byte vectors of O and of dO. The statistics rows that belong
// to no query (after each sequence's rows up to the next sequence's block, and
// to stat_rows at the end) get lse2 = -inf and delta = 0, so every row a tile
// can read is finite. Then the dQ accumulator is zeroed.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const PrepParams p) {
  using E = Elem<BF16>;
  constexpr int VPR = D / 8;                        // 16-byte vectors per row
  constexpr int G = VPR / 2 < 32 ? VPR / 2 : 32;    // lanes per item
  constexpr int PER = VPR / G;                      // vectors per lane (2 for D = 128, 256, 512)
  constexpr int PER_WARP = 32 / G;                  // items one warp handles per step
  const Geom& g = p.g;
  // THD metadata that failed the guard is not used for addressing
  if (p.guard && *reinterpret_cast<volatile const int*>(p.guard)) return;
  const int lane = threadIdx.x % 32;
  const int sub = lane % G;
  const long long items = (long long)g.rows_q * g.nh_q;
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long n_warps = (long long)gridDim.x * blockDim.x / 32;
  // Below head_dim 512, two items per lane group and step (U), their loads
  // issued together, so each thread keeps 4 * PER 16-byte loads in flight (at
  // 512 the doubled registers cost more occupancy than they gain). Warp-
  // uniform trip count, so the shuffles below always see all 32 lanes.
  constexpr int U = D < 512 ? 2 : 1;
  for (long long base = warp_id * PER_WARP * U; base < items; base += n_warps * PER_WARP * U) {
    uint4 a[U][PER], c[U][PER];
    long long its[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      its[u] = base + u * PER_WARP + lane / G;
      const uint4* o4 = reinterpret_cast<const uint4*>(p.o) + its[u] * VPR;
      const uint4* d4 = reinterpret_cast<const uint4*>(p.dout) + its[u] * VPR;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int v = 0; v < PER; ++v) {
        const bool live = its[u] < items;
        a[u][v] = live && SDPA_ADDR_OK(g.chk, o4 + sub + v * G, 16) ? o4[sub + v * G] : z;
        c[u][v] = live && SDPA_ADDR_OK(g.chk, d4 + sub + v * G, 16) ? d4[sub + v * G] : z;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float acc = 0.f;
#pragma unroll
      for (int v = 0; v < PER; ++v) {
        const uint32_t au[4] = {a[u][v].x, a[u][v].y, a[u][v].z, a[u][v].w};
        const uint32_t cu[4] = {c[u][v].x, c[u][v].y, c[u][v].z, c[u][v].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = E::unpack(au[e]), fc = E::unpack(cu[e]);
          acc = fmaf(fa.x, fc.x, acc);
          acc = fmaf(fa.y, fc.y, acc);
        }
      }
#pragma unroll
      for (int sh = G / 2; sh > 0; sh /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, sh, G);
      const long long it = its[u];
      if (it < items && sub == 0) {
        const int row = (int)(it / g.nh_q), hg = (int)(it - (long long)row * g.nh_q);
        const float l = SDPA_ADDR_OK(g.chk, p.lse + it, 4) ? p.lse[it] : -INFINITY;
        const long long st = (long long)hg * p.stat_rows + stat_row(g, row);
        if (SDPA_ADDR_OK(g.chk, p.delta + st, 4)) p.delta[st] = acc;
        if (SDPA_ADDR_OK(g.chk, p.lse2 + st, 4)) p.lse2[st] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
      }
    }
  }
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  // statistics rows of no query: per (sequence, generic head); SBHD keeps its
  // batches apart through the generic head, so it has one "sequence"
  const int nseq = g.layout == SDPA_SBHD ? 1 : g.batch;
  const int heads = g.layout == SDPA_SBHD ? g.nh_q : g.hq;
  for (long long it = tid; it < (long long)nseq * heads; it += nthreads) {
    const int b = (int)(it / heads), hg = (int)(it - (long long)b * heads);
    const SeqInfo si = seq_info(g, b);
    const int a = si.srow0 + si.lq;
    const int e = (b + 1 == nseq) ? p.stat_rows : seq_info(g, b + 1).srow0;
    for (int r = a; r < e; ++r) {
      const long long st = (long long)hg * p.stat_rows + r;
      if (SDPA_ADDR_OK(g.chk, p.delta + st, 4)) p.delta[st] = 0.f;
      if (SDPA_ADDR_OK(g.chk, p.lse2 + st, 4)) p.lse2[st] = -INFINITY;
    }
  }
  // zero the dQ accumulator
  const long long n4 = p.dq_acc ? (long long)g.nh_q * g.rows_q * g.d / 4 : 0;
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  constexpr int UZ = D < 512 ? 4 : 1;  // stores per thread and step (chosen by measurement, as U)
  for (long long it = tid; it < n4; it += UZ * nthreads) {
#pragma unroll
    for (int u = 0; u < UZ; ++u) {
      const long long x = it + u * nthreads;
      if (x < n4 && SDPA_ADDR_OK(g.chk, acc4 + x, 16)) acc4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// SMs of the current device (queried per call: a process may drive several GPUs).
static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0)
    n = 148;
  return n;
}

int launch_preprocess(const PrepParams& pp, bool bf16, cudaStream_t s) {
  if (pp.g.batch <= 0) return SDPA_OK;
  const unsigned grid = (unsigned)sm_count() * 8;  // 8 blocks of 256 threads per SM, grid-stride
  const int d = pp.g.d;
#define PREP(B, DD) preprocess_kernel<B, DD><<<grid, 256, 0, s>>>(pp)
  if (d == 128) { if (bf16) PREP(true, 128); else PREP(false, 128); }
  else if (d == 256) { if (bf16) PREP(true, 256); else PREP(false, 256); }
  else if (d == 512) { if (bf16) PREP(true, 512); else PREP(false, 512); }
  else return SDPA_ERR_UNSUPPORTED;
#undef PREP
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

// dq[(row*nh + head)*D + d] = scale * acc[(head*rows + row)*D + d]; each
// thread converts 8 consecutive columns.
template <bool BF16>
__global__ void __launch_bounds__(256) dq_finalize_kernel(const Geom g, const float* __restrict__ acc, void* dq,
                                                         const int* guard) {
  using E = Elem<BF16>;
  if (guard && *guard) return;
  const int d8 = g.d / 8;
  const long long n = (long long)g.nh_q * g.rows_q * d8;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < n; it += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(it % d8);
    const long long hr = it / d8;  // head * rows + row
    const int head = (int)(hr / g.rows_q), row = (int)(hr % g.rows_q);
    const float4* src = reinterpret_cast<const float4*>(acc + hr * g.d + c * 8);
    uint4* dst = reinterpret_cast<uint4*>(dq) + ((long long)row * g.nh_q + head) * d8 + c;
    if (!SDPA_ADDR_OK(g.chk, src, 32) || !SDPA_ADDR_OK(g.chk, dst, 16)) continue;
    const float4 a = src[0], b = src[1];
    uint4 out;
    out.x = E::pack(a.x * g.scale, a.y * g.scale);
    out.y = E::pack(a.z * g.scale, a.w * g.scale);
    out.z = E::pack(b.x * g.scale, b.y * g.scale);
    out.w = E::pack(b.z * g.scale, b.w * g.scale);
    *dst = out;
  }
}

int launch_dq_finalize(const Geom& g, const float* dq_acc, void* dq, const int* guard, bool bf16, cudaStream_t s) {
  const int grid = sm_count() * 8;
  if (bf16)
    dq_finalize_kernel<true><<<grid, 256, 0, s>>>(g, dq_acc, dq, guard);
  else
    dq_finalize_kernel<false><<<grid, 256, 0, s>>>(g, dq_acc, dq, guard);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

// Exercises the bounded wait every pipelined kernel uses: one thread waits on
// an mbarrier that nothing ever arrives on, gives up after `limit_ns`, and
// records SDPA_ERR_TIMEOUT exactly as a stalled kernel would.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit_ns)) record_error(err, SDPA_ERR_TIMEOUT);
}

int launch_wait_selftest(uint64_t limit_ns, int* err, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, err);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace sdpa
