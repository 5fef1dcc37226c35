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
// (d = 64) segments. The row's C lse values are read once, spread over its
// lanes (max and sum by shuffles), and the loads of 8 chunks at a time are
// issued before their accumulation; the first 8 go out before the lse
// reduction, which they do not depend on. One resident wave of warps walks the
// rows.
#include "common.cuh"
#include "kernels.h"

namespace eba {
namespace {

constexpr int kMergeThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int kLanesPerRow = D / 4;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kSlots = (ATTN_MAX_CHUNKS + kLanesPerRow - 1) / kLanesPerRow;  // lse values per lane
  const int lane = threadIdx.x & 31;
  const int seg = lane % kLanesPerRow;
  const int sub = lane / kLanesPerRow;  // row of the warp's group
  const long long n_warps = static_cast<long long>(gridDim.x) * (kMergeThreads / 32);
  const long long warp0 = (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) / 32;
  const int C = a.n_chunks;
  const long long o_stride = a.rows * D;
  // Grid-stride over groups of kRowsPerWarp rows: one resident wave of warps.
  for (long long grp = warp0; grp * kRowsPerWarp < a.rows; grp += n_warps) {
    const long long row = grp * kRowsPerWarp + sub;
    const bool valid = row < a.rows;
    const float* o_p = a.o_parts + row * D + seg * 4;
    // The first 8 partials do not depend on the weights: their loads go out
    // before the lse reduction, so the two memory latencies overlap.
    float4 v0[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v0[u] = (valid && u < C) ? __ldcs(reinterpret_cast<const float4*>(o_p + u * o_stride))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    // Chunk lse values: lane seg holds chunks seg, seg + kLanesPerRow, ... of
    // its row (each read once); max and sum by shuffles within the row's lanes.
    float l[kSlots], e[kSlots];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      const int cc = seg + k * kLanesPerRow;
      l[k] = (valid && cc < C) ? __ldg(a.lse_parts + row + static_cast<long long>(cc) * a.rows)
                               : -INFINITY;
      M = fmaxf(M, l[k]);
    }
#pragma unroll
    for (int m = kLanesPerRow / 2; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    const bool empty = (M == -INFINITY);
    const float Ms = empty ? 0.f : M;
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      e[k] = ex2_approx((l[k] - Ms) * kLog2e);
      tot += e[k];
    }
    // weight numerator of chunk cc, from the lane of this row that holds it
    auto ex_of = [&](int cc) {
      const int slot = cc / kLanesPerRow;
      float mine = e[0];
#pragma unroll
      for (int k = 1; k < kSlots; ++k) mine = (slot == k) ? e[k] : mine;
      return __shfl_sync(0xffffffffu, mine, sub * kLanesPerRow + cc % kLanesPerRow);
    };
#pragma unroll
    for (int m = kLanesPerRow / 2; m > 0; m >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, m);
    const float inv_tot = empty ? 0.f : 1.f / tot;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float w = ex_of(u) * inv_tot;  // 0 for u >= C (exp of -inf)
      acc.x = fmaf(w, v0[u].x, acc.x);
      acc.y = fmaf(w, v0[u].y, acc.y);
      acc.z = fmaf(w, v0[u].z, acc.z);
      acc.w = fmaf(w, v0[u].w, acc.w);
    }
    int c = 8;
    for (; c + 8 <= C; c += 8) {
      float4 v[8];
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int cu = c + u;
        w[u] = ex_of(cu) * inv_tot;
        v[u] = valid && !empty ? __ldcs(reinterpret_cast<const float4*>(o_p + cu * o_stride))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
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
      const float w = ex_of(c) * inv_tot;
      const float4 v = valid && !empty ? __ldcs(reinterpret_cast<const float4*>(o_p + c * o_stride))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (empty) acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
      uint2 packed = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o) + row * D + seg * 4) = packed;
      if (seg == 0) a.lse[row] = empty ? -INFINITY : M + lg2_approx(tot) * kLn2;
    }
  }
}

template <int D>
cudaError_t launch_merge_t(const MergeArgs& a, cudaStream_t stream) {
  constexpr int kRowsPerBlock = (kMergeThreads / 32) * (32 / (D / 4));
  const long long need = (a.rows + kRowsPerBlock - 1) / kRowsPerBlock;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, merge_kernel<D>, kMergeThreads, 0);
  if (e != cudaSuccess) return e;
  const long long wave = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
  const long long blocks = need < wave ? need : wave;
  return launch_pdl(merge_kernel<D>, dim3(static_cast<unsigned>(blocks)), dim3(kMergeThreads), 0,
                    stream, a);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, int d, cudaStream_t stream) {
  return d == 64 ? launch_merge_t<64>(a, stream) : launch_merge_t<128>(a, stream);
}

}  // namespace eba
