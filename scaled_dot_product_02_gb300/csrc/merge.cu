// merge.cu -- log-sum-exp merge of partial attention results over a split of
// the keys (the context-parallel LSE handling of TransformerEngine PR #3527
// and PR #3693, with neutral statistics for empty blocks):
//   LSE = ln sum_k exp(LSE_k),   O = sum_k exp(LSE_k - LSE) O_k
// per item (a row of one head). Memory-bound: each item reads n_parts
// 16-bit rows of D values and n_parts fp32 statistics and writes one row and
// one statistic; G lanes share an item, each owning 16-byte vectors of it.
#include <algorithm>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace sdpa {

namespace {

template <bool BF16, int D>
__global__ void __launch_bounds__(256) merge_kernel(const uint4* __restrict__ o_parts, const float* __restrict__ lse_parts,
                                                    uint4* __restrict__ o, float* __restrict__ lse, long long items,
                                                    int n_parts, AddrTable* chk) {
  // a part's LSE (an access the address check rejects reads as an empty part)
  auto part_lse = [&](int k, long long it) {
    const float* a = lse_parts + (long long)k * items + it;
    return SDPA_ADDR_OK(chk, a, 4) ? __ldg(a) : -INFINITY;
  };
  using E = Elem<BF16>;
  constexpr int VPR = D / 8;              // 16-byte vectors per row
  constexpr int G = VPR < 32 ? VPR : 32;  // lanes per item
  constexpr int PER = VPR / G;            // vectors per lane
  constexpr int PER_WARP = 32 / G;
  const int lane = threadIdx.x % 32;
  const int sub = lane % G;
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long n_warps = (long long)gridDim.x * blockDim.x / 32;
  for (long long base = warp_id * PER_WARP; base < items; base += n_warps * PER_WARP) {
    const long long it = base + lane / G;
    if (it >= items) continue;  // no shuffles below: lanes may leave independently
    float m = -INFINITY;
    for (int k = 0; k < n_parts; ++k) m = fmaxf(m, part_lse(k, it));
    float acc[PER][8];
#pragma unroll
    for (int v = 0; v < PER; ++v)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[v][e] = 0.f;
    float l = -INFINITY;
    if (m != -INFINITY) {
      float s = 0.f;
      for (int k = 0; k < n_parts; ++k) s += expf(part_lse(k, it) - m);
      l = m + logf(s);
#pragma unroll 4
      for (int k = 0; k < n_parts; ++k) {
        const float lk = part_lse(k, it);
        // an empty block (LSE -inf) is skipped, not weighted by 0, so whatever
        // its rows hold stays out of the sum
        if (lk == -INFINITY) continue;
        const float w = expf(lk - l);
        const uint4* src = o_parts + ((long long)k * items + it) * VPR;
#pragma unroll
        for (int v = 0; v < PER; ++v) {
          const uint4 x = SDPA_ADDR_OK(chk, src + sub + v * G, 16) ? __ldg(src + sub + v * G) : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = E::unpack(u[e]);
            acc[v][2 * e] = fmaf(w, f.x, acc[v][2 * e]);
            acc[v][2 * e + 1] = fmaf(w, f.y, acc[v][2 * e + 1]);
          }
        }
      }
    }
    uint4* dst = o + it * VPR;
#pragma unroll
    for (int v = 0; v < PER; ++v)
      if (SDPA_ADDR_OK(chk, dst + sub + v * G, 16))
        dst[sub + v * G] = make_uint4(E::pack(acc[v][0], acc[v][1]), E::pack(acc[v][2], acc[v][3]),
                                    E::pack(acc[v][4], acc[v][5]), E::pack(acc[v][6], acc[v][7]));
    if (sub == 0 && SDPA_ADDR_OK(chk, lse + it, 4)) lse[it] = l;
  }
}

template <bool BF16, int D>
int launch_merge_t(const void* o_parts, const float* lse_parts, void* o, float* lse, long long items, int n_parts,
                   AddrTable* chk, cudaStream_t s) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDPA_ERR_CUDA;
  constexpr int G = (D / 8) < 32 ? (D / 8) : 32;
  const long long warps_needed = (items + (32 / G) - 1) / (32 / G);
  const long long blocks = std::min<long long>((warps_needed + 7) / 8, (long long)sms * 8);
  merge_kernel<BF16, D><<<(unsigned)std::max<long long>(blocks, 1), 256, 0, s>>>(
      static_cast<const uint4*>(o_parts), lse_parts, static_cast<uint4*>(o), lse, items, n_parts, chk);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace

int launch_merge(const void* o_parts, const float* lse_parts, void* o, float* lse, long long items, int head_dim,
                 int n_parts, bool bf16, AddrTable* chk, cudaStream_t s) {
  if (items == 0) return SDPA_OK;
#define MERGE(B, DD) return launch_merge_t<B, DD>(o_parts, lse_parts, o, lse, items, n_parts, chk, s)
  if (head_dim == 128) { if (bf16) MERGE(true, 128); MERGE(false, 128); }
  if (head_dim == 256) { if (bf16) MERGE(true, 256); MERGE(false, 256); }
  if (head_dim == 512) { if (bf16) MERGE(true, 512); MERGE(false, 512); }
#undef MERGE
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace sdpa
