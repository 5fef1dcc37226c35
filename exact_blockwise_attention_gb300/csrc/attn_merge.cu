// Exact merge of split-KV partial attention results ("LV-XAttn", ICML 2025
// poster, Abstract and Lay Summary: the key/value blocks stay in place and the
// split attention is exact, so merging partials reproduces the unsplit output).
//
// Per output row, over the C chunks:
//   M = max_c lse_c,  tot = sum_c exp(lse_c - M),  lse = M + ln tot,
//   O = sum_c (exp(lse_c - M) / tot) * O_c   -> bf16.
// A row whose chunks all have lse_c = -inf gets O = 0, lse = -inf.
//
// Memory-bound: each row reads C fp32 vectors of d elements and writes one bf16
// vector. d/4 lanes share a row, each lane owning 16 bytes of every partial, so
// a warp's loads of one partial are contiguous 512-byte (d = 128) or 2 x 256-byte
// (d = 64) segments. Loads of all chunks are issued before the accumulation so
// C independent requests per lane are in flight.
#include "common.cuh"
#include "kernels.h"

namespace eba {
namespace {

constexpr int kMergeThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  constexpr int kLanesPerRow = D / 4;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const long long gwarp =
      (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  const long long row = gwarp * kRowsPerWarp + lane / kLanesPerRow;
  const int seg = lane % kLanesPerRow;
  if (row >= a.rows) return;
  const int C = a.n_chunks;
  const float* lse_p = a.lse_parts + row;
  const float* o_p = a.o_parts + row * D + seg * 4;
  const long long o_stride = a.rows * D;

  float M = -INFINITY;
  for (int c = 0; c < C; ++c) M = fmaxf(M, __ldg(lse_p + c * a.rows));

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse_out = -INFINITY;
  if (M != -INFINITY) {
    float tot = 0.f;
    for (int c = 0; c < C; ++c) tot += ex2_approx((__ldg(lse_p + c * a.rows) - M) * kLog2e);
    const float inv_tot = 1.f / tot;
    int c = 0;
    for (; c + 8 <= C; c += 8) {
      float4 v[8];
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        v[u] = __ldcs(reinterpret_cast<const float4*>(o_p + (c + u) * o_stride));
        w[u] = ex2_approx((__ldg(lse_p + (c + u) * a.rows) - M) * kLog2e) * inv_tot;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x = fmaf(w[u], v[u].x, acc.x);
        acc.y = fmaf(w[u], v[u].y, acc.y);
        acc.z = fmaf(w[u], v[u].z, acc.z);
        acc.w = fmaf(w[u], v[u].w, acc.w);
      }
    }
    for (; c < C; ++c) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(o_p + c * o_stride));
      const float w = ex2_approx((__ldg(lse_p + c * a.rows) - M) * kLog2e) * inv_tot;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    lse_out = M + lg2_approx(tot) * kLn2;
  }
  uint2 packed = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o) + row * D + seg * 4) = packed;
  if (seg == 0) a.lse[row] = lse_out;
}

template <int D>
cudaError_t launch_merge_t(const MergeArgs& a, cudaStream_t stream) {
  constexpr int kRowsPerBlock = (kMergeThreads / 32) * (32 / (D / 4));
  const long long blocks = (a.rows + kRowsPerBlock - 1) / kRowsPerBlock;
  merge_kernel<D><<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, int d, cudaStream_t stream) {
  return d == 64 ? launch_merge_t<64>(a, stream) : launch_merge_t<128>(a, stream);
}

}  // namespace eba
