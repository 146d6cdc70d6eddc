// aux.cu -- the memory-bound steps around the attention kernels:
//   * the THD metadata guard (TransformerEngine PR #3705, "Execution and
//     supported scope": compactness is checked on the GPU on every
//     execution -- zero-based cumulative lengths, valid bounds, non-empty KV
//     for live Q);
//   * the backward preprocess: delta = rowsum(dO * O) in fp32, -LSE*log2(e)
//     (-inf for rows without keys), and the fp32 dQ accumulator zeroed;
//   * the dQ finalise: dQ = scale * accumulator, cast to the input dtype.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

__global__ void guard_kernel(const int32_t* cu_q, const int32_t* cu_kv, int batch, int total_q, int total_kv,
                             int max_q, int max_kv, int* guard, int* err) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = (cu_q[0] != 0) || (cu_kv[0] != 0) || (cu_q[batch] != total_q) || (cu_kv[batch] != total_kv);
  __syncthreads();
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    const int lq = cu_q[b + 1] - cu_q[b];
    const int lk = cu_kv[b + 1] - cu_kv[b];
    if (lq < 0 || lk < 0 || lq > max_q || lk > max_kv || (lq > 0 && lk == 0)) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *guard = bad ? SDPA_ERR_BAD_SEQLENS : 0;
    if (bad) record_error(err, SDPA_ERR_BAD_SEQLENS);
  }
}

int launch_guard(const Geom& g, int total_q, int total_kv, int* guard, int* err, cudaStream_t s) {
  guard_kernel<<<1, 256, 0, s>>>(g.cu_q, g.cu_kv, g.batch, total_q, total_kv, g.sq, g.sk, guard, err);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

// One group of G lanes per (row, head) item; each lane owns D/(8G) 16-byte
// vectors of O and dO.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const PrepParams p) {
  using E = Elem<BF16>;
  constexpr int VPR = D / 8;                 // 16-byte vectors per row
  constexpr int G = VPR < 32 ? VPR : 32;     // lanes per item
  constexpr int PER = VPR / G;               // vectors per lane
  const Geom& g = p.g;
  const int lane = threadIdx.x % 32;
  const int sub = lane % G;
  constexpr int PER_WARP = 32 / G;  // items one warp handles per step
  const long long items = (long long)g.rows_q * g.nh_q;
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long n_warps = (long long)gridDim.x * blockDim.x / 32;
  // warp-uniform trip count, so the shuffles below always see all 32 lanes
  for (long long base = warp_id * PER_WARP; base < items; base += n_warps * PER_WARP) {
    const long long it = base + lane / G;
    const bool live = it < items;
    float acc = 0.f;
    if (live) {
      const uint4* o4 = reinterpret_cast<const uint4*>(p.o) + it * VPR;
      const uint4* d4 = reinterpret_cast<const uint4*>(p.dout) + it * VPR;
#pragma unroll
      for (int v = 0; v < PER; ++v) {
        const uint4 a = o4[sub + v * G], b = d4[sub + v * G];
        const uint32_t au[4] = {a.x, a.y, a.z, a.w}, bu[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = E::unpack(au[e]), fb = E::unpack(bu[e]);
          acc = fmaf(fa.x, fb.x, acc);
          acc = fmaf(fa.y, fb.y, acc);
        }
      }
    }
#pragma unroll
    for (int sh = G / 2; sh > 0; sh /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, sh, G);
    if (live && sub == 0) {
      const int row = (int)(it / g.nh_q), head = (int)(it % g.nh_q);
      const float l = p.lse[(long long)row * g.nh_q + head];
      const long long si = (long long)head * p.stat_rows + row;
      p.delta[si] = acc;
      p.lse2[si] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
    }
  }
  // padding rows of the statistics, read by tiles that overhang the end
  const long long pad_items = (long long)g.nh_q * (p.stat_rows - g.rows_q);
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < pad_items;
       it += (long long)gridDim.x * blockDim.x) {
    const int head = (int)(it / (p.stat_rows - g.rows_q));
    const int row = g.rows_q + (int)(it % (p.stat_rows - g.rows_q));
    p.delta[(long long)head * p.stat_rows + row] = 0.f;
    p.lse2[(long long)head * p.stat_rows + row] = -INFINITY;
  }
  // zero the dQ accumulator
  const long long n4 = p.dq_acc ? (long long)g.nh_q * g.rows_q * g.d / 4 : 0;
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < n4; it += (long long)gridDim.x * blockDim.x)
    acc4[it] = make_float4(0.f, 0.f, 0.f, 0.f);
}

static int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

int launch_preprocess(const PrepParams& pp, bool bf16, cudaStream_t s) {
  const int grid = sm_count() * 8;
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
    const float4 a = src[0], b = src[1];
    uint4 out;
    out.x = E::pack(a.x * g.scale, a.y * g.scale);
    out.y = E::pack(a.z * g.scale, a.w * g.scale);
    out.z = E::pack(b.x * g.scale, b.y * g.scale);
    out.w = E::pack(b.z * g.scale, b.w * g.scale);
    reinterpret_cast<uint4*>(dq)[((long long)row * g.nh_q + head) * d8 + c] = out;
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
