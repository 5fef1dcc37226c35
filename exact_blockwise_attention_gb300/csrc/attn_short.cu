// Forward attention over very short sequences (at most 8 queries and 8 keys
// per (batch, head)) on the CUDA cores.
//
// Factorised video attention has a temporal pass whose sequences are the few
// frames of one spatial position ("Training a Large Video Model on a Single
// Machine in a Day", §3 and §4.1 "Discussion": attention factorised over
// space and time). There every (batch, head) is a tiny independent problem:
// S = scale Q K^T is at most 8 x 8, and the whole computation is a few
// kilobytes of HBM per sequence against a few thousand multiply-adds. The
// 128-row tensor-core tiles would spend a full pipeline round (loads, two
// MMA hand-offs, epilogue) on each such block, so this path is HBM-bound by
// design instead: the arithmetic is cheap next to the bytes.
//
// Same result as the tiled forward, O = softmax(scale Q K^T) V and the
// natural-log lse per query row, with P kept in fp32 (not rounded to bf16
// before P V).
//
// One warp per sequence, walking the sequences with a persistent grid:
//   - loads: a sequence's Q, K and V are three contiguous blocks, staged by
//     three 1-D TMA bulk copies into the warp's shared-memory double buffer
//     (completion on an mbarrier), the next sequence's issued before this
//     one is computed, so that its bytes stream in meanwhile;
//   - from there every lane reads only its own slices once (the products
//     work in registers: warp-wide 16-byte shared loads cost four wavefronts
//     each, which made a version reading whole rows from shared memory bound
//     by the shared-memory pipe). Lane = 16 a + 8 b + s:
//   - scores: lane (a, b, s) holds query rows 4a..4a+3 and key rows 4b..4b+3,
//     columns [s D/8, (s+1) D/8) of each, and forms the 4 x 4 partial dot
//     products over its columns (two-lane packed
//     fp32 FMAs); a three-level transpose-reduce over s (shuffles) leaves
//     each lane two whole scores, row 4a + s/2, keys 4b + 2 (s & 1) + {0, 1};
//   - softmax: a row's eight scores sit in four lanes (lane bits 0 and 3),
//     so its max and sum take two shuffles each; P stays fp32;
//   - P V: the 16 lanes of row group a gather its 32 weights by shuffles;
//     lane (a, b, s) owns columns [t D/16, (t+1) D/16), t = 8b + s, of rows
//     4a..4a+3, with those columns of every V row in registers; O leaves as
//     bf16, 128 or 256 contiguous bytes per row.
#include "common.cuh"
#include "kernels.h"

namespace eba {
namespace {

constexpr int kShortThreads = 128;
constexpr int kShortWarps = kShortThreads / 32;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float2 bf16x2_f32(uint32_t w) {
  return make_float2(bf16lo_f32(w), bf16hi_f32(w));
}

// One warp's double buffer: per buffer, Q, K and V of one sequence (at most
// 8 rows each, bf16); then two mbarriers per warp and the block's abort flag.
template <int D>
struct ShortSmem {
  static constexpr int kTile = kShortMax * D * 2;
  static constexpr int kBuf = 3 * kTile;
  static constexpr int kWarp = 2 * kBuf;
  static constexpr int offBar = kShortWarps * kWarp;
  static constexpr int offAbort = offBar + kShortWarps * 16;
  static constexpr int kBytes = offAbort + 16;
};

// W bf16 values (W = 8 or 16) from shared memory as W / 2 packed words (zero
// for rows past the sequence: the buffer still holds an earlier sequence there).
template <int W>
__device__ __forceinline__ void lds_words(uint32_t (&w)[W / 2], const uint8_t* p, bool ok) {
#pragma unroll
  for (int h = 0; h < W / 8; ++h) {
    const uint4 x = ok ? reinterpret_cast<const uint4*>(p)[h] : make_uint4(0u, 0u, 0u, 0u);
    w[4 * h] = x.x;
    w[4 * h + 1] = x.y;
    w[4 * h + 2] = x.z;
    w[4 * h + 3] = x.w;
  }
}

template <int D>
__global__ void __launch_bounds__(kShortThreads) fwd_short_kernel(const ShortArgs a) {
  constexpr int W = D / 8;    // score columns per lane
  constexpr int CW = D / 16;  // output columns per lane
  using S = ShortSmem<D>;
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(128) uint8_t short_smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ga = lane >> 4, gb = (lane >> 3) & 1, gs = lane & 7;
  const int t = lane & 15;  // output column block within the row group
  const int Lq = a.Lq, Lk = a.Lk;
  const float sl2 = a.scale_log2;
  const __nv_bfloat16* const q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* const k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* const v = static_cast<const __nv_bfloat16*>(a.v);
  __nv_bfloat16* const o = static_cast<__nv_bfloat16*>(a.o);
  const unsigned full = 0xffffffffu;
  // this lane's two scores: row 4a + s/2, keys 4b + 2 (s & 1) + {0, 1}
  const int my_row = 4 * ga + (gs >> 1);
  const int my_key = 4 * gb + 2 * (gs & 1);

  uint8_t* const wbuf = short_smem + warp * S::kWarp;
  const uint32_t bar = smem_u32(short_smem + S::offBar + warp * 16);  // + 8 b: buffer b full
  volatile int* abort_flag = reinterpret_cast<volatile int*>(short_smem + S::offAbort);
  const DeviceStatus st{a.status, a.limit_ns};
  if (threadIdx.x == 0) *abort_flag = 0;
  if (lane == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 8, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t q_bytes = static_cast<uint32_t>(Lq) * D * 2, k_bytes = static_cast<uint32_t>(Lk) * D * 2;
  auto issue = [&](long long seq, int b) {  // lane 0: Q, K, V of `seq` into buffer b
    const uint32_t dst = smem_u32(wbuf + b * S::kBuf);
    mbar_arrive_expect_tx(bar + 8 * b, q_bytes + 2 * k_bytes);
    bulk_load(dst, q + seq * Lq * D, q_bytes, bar + 8 * b);
    bulk_load(dst + S::kTile, k + seq * Lk * D, k_bytes, bar + 8 * b);
    bulk_load(dst + 2 * S::kTile, v + seq * Lk * D, k_bytes, bar + 8 * b);
  };

  const long long n_warps = static_cast<long long>(gridDim.x) * kShortWarps;
  long long seq = static_cast<long long>(blockIdx.x) * kShortWarps + warp;
  int n = 0;  // this warp's iteration: buffer n % 2, its (n / 2)-th use
  bool ok = true;
  if (seq < a.n_seq && lane == 0) issue(seq, 0);
  for (; seq < a.n_seq; seq += n_warps, ++n) {
    const int b = n & 1;
    if (seq + n_warps < a.n_seq && lane == 0) issue(seq + n_warps, b ^ 1);
    if (!(ok = __all_sync(full, mbar_wait(bar + 8 * b, (n >> 1) & 1, abort_flag, st)))) break;
    const uint8_t* sq = wbuf + b * S::kBuf;
    const uint8_t* sk = sq + S::kTile;
    const uint8_t* sv = sq + 2 * S::kTile;
    // ---- this lane's Q, K column slices for the scores, V column block for P V
    uint32_t qw[4][W / 2], kw[4][W / 2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      lds_words<W>(qw[r], sq + ((4 * ga + r) * D + gs * W) * 2, 4 * ga + r < Lq);
      lds_words<W>(kw[r], sk + ((4 * gb + r) * D + gs * W) * 2, 4 * gb + r < Lk);
    }
    uint32_t vw[8][CW / 2];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint8_t* vp = sv + (j * D + t * CW) * 2;
      if constexpr (CW == 4) {
        const uint2 x = j < Lk ? *reinterpret_cast<const uint2*>(vp) : make_uint2(0u, 0u);
        vw[j][0] = x.x;
        vw[j][1] = x.y;
      } else {
        const uint4 x = j < Lk ? *reinterpret_cast<const uint4*>(vp) : make_uint4(0u, 0u, 0u, 0u);
        vw[j][0] = x.x;
        vw[j][1] = x.y;
        vw[j][2] = x.z;
        vw[j][3] = x.w;
      }
    }
    __syncwarp();  // buffer b is free for the sequence after next

    // ---- partial scores over this lane's columns: sp[r][c] = q_r . k_c
    float2 acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < W / 2; ++h) {
      float2 qf[4], kf[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        qf[r] = bf16x2_f32(qw[r][h]);
        kf[r] = bf16x2_f32(kw[r][h]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fma2(qf[r], kf[c], acc[r][c]);
    }
    float v16[16];  // index r * 4 + c
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) v16[r * 4 + c] = acc[r][c].x + acc[r][c].y;

    // ---- transpose-reduce over s: split on r1 (lane bit 2), r0 (bit 1), c1 (bit 0)
    float v8[8], v4[4], sc[2];
    {
      const bool hi = (gs >> 2) & 1;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float send = hi ? v16[u] : v16[8 + u];
        v8[u] = (hi ? v16[8 + u] : v16[u]) + __shfl_xor_sync(full, send, 4);
      }
    }
    {
      const bool hi = (gs >> 1) & 1;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float send = hi ? v8[u] : v8[4 + u];
        v4[u] = (hi ? v8[4 + u] : v8[u]) + __shfl_xor_sync(full, send, 2);
      }
    }
    {
      const bool hi = gs & 1;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float send = hi ? v4[u] : v4[2 + u];
        sc[u] = (hi ? v4[2 + u] : v4[u]) + __shfl_xor_sync(full, send, 1);
      }
    }

    // ---- softmax of row my_row (four lanes: bits 0 and 3), base 2
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (my_key + u >= Lk) sc[u] = -INFINITY;
    float m = fmaxf(sc[0], sc[1]);
    m = fmaxf(m, __shfl_xor_sync(full, m, 1));
    m = fmaxf(m, __shfl_xor_sync(full, m, 8));
    const float m2 = m * sl2;
    float p[2];
    p[0] = ex2_approx(fmaf(sc[0], sl2, -m2));
    p[1] = ex2_approx(fmaf(sc[1], sl2, -m2));
    float l = p[0] + p[1];
    l += __shfl_xor_sync(full, l, 1);
    l += __shfl_xor_sync(full, l, 8);
    if ((lane & 9) == 0 && my_row < Lq) a.lse[seq * Lq + my_row] = (m2 + lg2_approx(l)) * kLn2;
    const float inv_l = 1.f / l;

    // ---- P V: gather the row group's 32 weights, then this lane's columns
    float pr[4][8];
#pragma unroll
    for (int src = 0; src < 16; ++src)
#pragma unroll
      for (int u = 0; u < 2; ++u)
        pr[(src & 7) >> 1][4 * (src >> 3) + 2 * (src & 1) + u] = __shfl_sync(full, p[u], src, 16);
    float inv[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) inv[r] = __shfl_sync(full, inv_l, 2 * r, 16);
    float2 oacc[4][CW / 2];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int h = 0; h < CW / 2; ++h) oacc[r][h] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float2 vf[CW / 2];
#pragma unroll
      for (int h = 0; h < CW / 2; ++h) vf[h] = bf16x2_f32(vw[j][h]);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int h = 0; h < CW / 2; ++h)
          oacc[r][h] = fma2(make_float2(pr[r][j], pr[r][j]), vf[h], oacc[r][h]);
    }
    __nv_bfloat16* os = o + (seq * Lq + 4 * ga) * D + t * CW;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (4 * ga + r < Lq) {
        uint32_t w[CW / 2];
#pragma unroll
        for (int h = 0; h < CW / 2; ++h) w[h] = pack_bf16(oacc[r][h].x * inv[r], oacc[r][h].y * inv[r]);
        if constexpr (CW == 4)
          *reinterpret_cast<uint2*>(os + r * D) = make_uint2(w[0], w[1]);
        else
          *reinterpret_cast<uint4*>(os + r * D) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (!ok && lane == 0) {
    // A wait gave up: the copies already issued (this iteration's and the
    // next one's) land before the block exits.
    mbar_wait_drain(bar + 8 * (n & 1), (n >> 1) & 1, st);
    if (seq + n_warps < a.n_seq) mbar_wait_drain(bar + 8 * ((n + 1) & 1), ((n + 1) >> 1) & 1, st);
  }
}

template <int D>
cudaError_t launch_short_t(const ShortArgs& a, cudaStream_t stream) {
  using S = ShortSmem<D>;
  auto kern = fwd_short_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kShortThreads, S::kBytes);
  if (e != cudaSuccess) return e;
  const long long need = (a.n_seq + kShortWarps - 1) / kShortWarps;
  const long long wave = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
  const long long blocks = need < wave ? need : wave;
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kShortThreads), S::kBytes,
                    stream, a);
}

}  // namespace

cudaError_t launch_fwd_short(const ShortArgs& a, int d, cudaStream_t stream) {
  return d == 64 ? launch_short_t<64>(a, stream) : launch_short_t<128>(a, stream);
}

}  // namespace eba
