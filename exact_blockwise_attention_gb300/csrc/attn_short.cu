// Attention over very short sequences (at most 8 queries and 8 keys per
// (batch, head)) on the CUDA cores: forward and backward.
//
// Factorised video attention has a temporal pass whose sequences are the few
// frames of one spatial position ("Training a Large Video Model on a Single
// Machine in a Day", §3 and §4.1 "Discussion": attention factorised over
// space and time). There every (batch, head) is a tiny independent problem:
// S = scale Q K^T is at most 8 x 8, and the whole computation is a few
// kilobytes of HBM per sequence against a few thousand multiply-adds. The
// 128-row tensor-core tiles would spend a full pipeline round (loads, MMA
// hand-offs, epilogue) on each such block, so this path is HBM-bound by design
// instead: the arithmetic is cheap next to the bytes.
//
// Same results as the tiled kernels, computed with P in fp32 (not rounded to
// bf16):
//   forward   O = softmax(scale Q K^T) V and the natural-log lse per row;
//   backward  P = exp(scale Q K^T - lse), dP = dO V^T,
//             D_i = sum_j P_ij dP_ij (equal to sum_k dO_ik O_ik, the row term
//             of the softmax Jacobian; formed from P and dP here, so O is not
//             read), dS = P * (dP - D), dV = P^T dO, dQ = scale dS K,
//             dK = scale dS^T Q.
//
// One warp per sequence, walking the sequences with a persistent grid:
//   - loads: each of a sequence's tensors is one contiguous block, staged by
//     a 1-D TMA bulk copy into the warp's shared-memory double buffer
//     (completion on an mbarrier, bounded wait); the next sequence's copies
//     are issued before this one is computed, so that its bytes stream in
//     meanwhile;
//   - from there every lane reads only its own slices (the products work in
//     registers: warp-wide 16-byte shared loads cost four wavefronts each,
//     which made a version reading whole rows from shared memory bound by the
//     shared-memory pipe). Lane = 16 a + 8 b + s:
//   - scores (S, and dP in the backward): lane (a, b, s) holds rows 4a..4a+3
//     of the query-side operand and rows 4b..4b+3 of the key-side one,
//     columns [s D/8, (s+1) D/8) of each, and forms the 4 x 4 partial dot
//     products over its columns (two-lane packed fp32 FMAs); a three-level
//     transpose-reduce over s (shuffles) leaves each lane two whole scores,
//     row 4a + s/2, keys 4b + 2 (s & 1) + {0, 1};
//   - a row's eight scores sit in four lanes (lane bits 0 and 3), so row
//     reductions (max, sum, D) take two shuffles each;
//   - products with a query-row block (P V, dS K): the 16 lanes of row group
//     a gather its 32 weights by shuffles; lane (a, b, s) owns columns
//     [t D/16, (t+1) D/16), t = 8b + s, of query rows 4a..4a+3;
//   - products with a key-row block (P^T dO, dS^T Q): lane (a, b, s) owns
//     those columns of key rows 4a..4a+3, gathering the 32 weights of that
//     key group from both row groups;
//   - outputs leave as bf16 rows, 128 or 256 contiguous bytes per warp row.
#include "common.cuh"
#include "kernels.h"

namespace eba {
namespace {

constexpr int kShortThreads = 128;
constexpr int kShortWarps = kShortThreads / 32;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

// One warp's double buffer: per buffer, NT tensors of one sequence (at most
// 8 rows each, bf16); then two mbarriers per warp and the block's abort flag.
template <int D, int NT>
struct ShortSmem {
  static constexpr int kTile = kShortMax * D * 2;
  static constexpr int kBuf = NT * kTile;
  static constexpr int kWarp = 2 * kBuf;
  static constexpr int offBar = kShortWarps * kWarp;
  static constexpr int offAbort = offBar + kShortWarps * 16;
  static constexpr int kBytes = offAbort + 16;
};

__device__ __forceinline__ float2 bf16x2_f32(uint32_t w) {
  return make_float2(bf16lo_f32(w), bf16hi_f32(w));
}

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

// This lane's two entries of X Y^T for row tiles X (nx rows) and Y (ny rows)
// in shared memory: row 4a + s/2, columns 4b + 2 (s & 1) + {0, 1}.
template <int D>
__device__ __forceinline__ void block_scores(const uint8_t* xs, const uint8_t* ys, int nx, int ny,
                                             int ga, int gb, int gs, float (&out)[2]) {
  constexpr int W = D / 8;  // columns per lane
  uint32_t xw[4][W / 2], yw[4][W / 2];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    lds_words<W>(xw[r], xs + ((4 * ga + r) * D + gs * W) * 2, 4 * ga + r < nx);
    lds_words<W>(yw[r], ys + ((4 * gb + r) * D + gs * W) * 2, 4 * gb + r < ny);
  }
  float2 acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = make_float2(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < W / 2; ++h) {
    float2 xf[4], yf[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      xf[r] = bf16x2_f32(xw[r][h]);
      yf[r] = bf16x2_f32(yw[r][h]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = fma2(xf[r], yf[c], acc[r][c]);
  }
  float v16[16];  // index r * 4 + c
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) v16[r * 4 + c] = acc[r][c].x + acc[r][c].y;
  // transpose-reduce over s: split on r1 (lane bit 2), r0 (bit 1), c1 (bit 0)
  float v8[8], v4[4];
  {
    const bool hi = (gs >> 2) & 1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float send = hi ? v16[u] : v16[8 + u];
      v8[u] = (hi ? v16[8 + u] : v16[u]) + __shfl_xor_sync(kFull, send, 4);
    }
  }
  {
    const bool hi = (gs >> 1) & 1;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float send = hi ? v8[u] : v8[4 + u];
      v4[u] = (hi ? v8[4 + u] : v8[u]) + __shfl_xor_sync(kFull, send, 2);
    }
  }
  {
    const bool hi = gs & 1;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float send = hi ? v4[u] : v4[2 + u];
      out[u] = (hi ? v4[2 + u] : v4[u]) + __shfl_xor_sync(kFull, send, 1);
    }
  }
}

// Columns [t D/16, (t+1) D/16) of rows 0..7 of a tile (n rows) in shared
// memory, as packed bf16 words (zero past row n).
template <int D>
__device__ __forceinline__ void load_cols(uint32_t (&c)[8][D / 32], const uint8_t* tile, int n,
                                          int t) {
  constexpr int CW = D / 16;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint8_t* p = tile + (j * D + t * CW) * 2;
    if constexpr (CW == 4) {
      const uint2 x = j < n ? *reinterpret_cast<const uint2*>(p) : make_uint2(0u, 0u);
      c[j][0] = x.x;
      c[j][1] = x.y;
    } else {
      const uint4 x = j < n ? *reinterpret_cast<const uint4*>(p) : make_uint4(0u, 0u, 0u, 0u);
      c[j][0] = x.x;
      c[j][1] = x.y;
      c[j][2] = x.z;
      c[j][3] = x.w;
    }
  }
}

// The 32 weights of this lane's query-row group (rows 4a..4a+3, all 8 keys),
// from the 16 lanes of its half-warp that hold them (two each).
__device__ __forceinline__ void gather_rows(float (&w)[4][8], const float (&x)[2]) {
#pragma unroll
  for (int src = 0; src < 16; ++src)
#pragma unroll
    for (int u = 0; u < 2; ++u)
      w[(src & 7) >> 1][4 * (src >> 3) + 2 * (src & 1) + u] = __shfl_sync(kFull, x[u], src, 16);
}

// The 32 weights of key group g (all 8 query rows, keys 4g..4g+3), w[c][i]
// for key 4g + c and row i, from the lanes of both row groups that hold them.
__device__ __forceinline__ void gather_keys(float (&w)[4][8], const float (&x)[2], int g) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int src = 16 * (i >> 2) + 8 * g + 2 * (i & 3) + ch;
#pragma unroll
      for (int u = 0; u < 2; ++u) w[2 * ch + u][i] = __shfl_sync(kFull, x[u], src);
    }
}

// Rows r0 + r (r < 4) of W C over this lane's columns: out_r = mul_r *
// sum_j w[r][j] cols[j], stored as bf16 at row0 + r D for rows below n.
template <int D>
__device__ __forceinline__ void product_store(const float (&w)[4][8],
                                              const uint32_t (&cols)[8][D / 32],
                                              const float (&mul)[4], __nv_bfloat16* row0, int r0,
                                              int n) {
  constexpr int CW = D / 16;
  float2 acc[4][CW / 2];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int h = 0; h < CW / 2; ++h) acc[r][h] = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float2 cf[CW / 2];
#pragma unroll
    for (int h = 0; h < CW / 2; ++h) cf[h] = bf16x2_f32(cols[j][h]);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int h = 0; h < CW / 2; ++h) acc[r][h] = fma2(make_float2(w[r][j], w[r][j]), cf[h], acc[r][h]);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    if (r0 + r < n) {
      uint32_t o[CW / 2];
#pragma unroll
      for (int h = 0; h < CW / 2; ++h) o[h] = pack_bf16(acc[r][h].x * mul[r], acc[r][h].y * mul[r]);
      if constexpr (CW == 4)
        *reinterpret_cast<uint2*>(row0 + r * D) = make_uint2(o[0], o[1]);
      else
        *reinterpret_cast<uint4*>(row0 + r * D) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// The warp's double-buffered staging: buffer n % 2 holds the NT tensors of
// the warp's n-th sequence.
template <int D, int NT>
struct ShortPipe {
  using S = ShortSmem<D, NT>;
  uint8_t* wbuf;
  uint32_t bar;  // + 8 b: buffer b full
  volatile int* abort_flag;
  DeviceStatus st;

  __device__ __forceinline__ ShortPipe(uint8_t* smem, int warp, int lane, int* status,
                                       unsigned long long limit)
      : wbuf(smem + warp * S::kWarp),
        bar(smem_u32(smem + S::offBar + warp * 16)),
        abort_flag(reinterpret_cast<volatile int*>(smem + S::offAbort)),
        st{status, limit} {
    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0) {
      mbar_init(bar, 1);
      mbar_init(bar + 8, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
  // lane 0: block i of src[i], bytes[i] long, into tile i of buffer b
  __device__ __forceinline__ void issue(int b, const void* const (&src)[NT],
                                        const uint32_t (&bytes)[NT]) {
    uint32_t total = 0;
#pragma unroll
    for (int i = 0; i < NT; ++i) total += bytes[i];
    const uint32_t dst = smem_u32(wbuf + b * S::kBuf);
    mbar_arrive_expect_tx(bar + 8 * b, total);
#pragma unroll
    for (int i = 0; i < NT; ++i) bulk_load(dst + i * S::kTile, src[i], bytes[i], bar + 8 * b);
  }
  // Iteration n's tensors have landed (false: a wait gave up).
  __device__ __forceinline__ bool wait(int n) {
    return __all_sync(kFull, mbar_wait(bar + 8 * (n & 1), (n >> 1) & 1, abort_flag, st));
  }
  __device__ __forceinline__ const uint8_t* tile(int n, int i) const {
    return wbuf + (n & 1) * S::kBuf + i * S::kTile;
  }
  // After a wait gave up at iteration n: the copies already issued (this
  // iteration's and, if `next`, the next one's) land before the block exits.
  __device__ __forceinline__ void drain(int n, bool next, int lane) {
    if (lane != 0) return;
    mbar_wait_drain(bar + 8 * (n & 1), (n >> 1) & 1, st);
    if (next) mbar_wait_drain(bar + 8 * ((n + 1) & 1), ((n + 1) >> 1) & 1, st);
  }
};

template <int D>
__global__ void __launch_bounds__(kShortThreads) fwd_short_kernel(const ShortArgs a) {
  constexpr int CW = D / 16;  // output columns per lane
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
  // this lane's two scores: row 4a + s/2, keys 4b + 2 (s & 1) + {0, 1}
  const int my_row = 4 * ga + (gs >> 1);
  const int my_key = 4 * gb + 2 * (gs & 1);
  ShortPipe<D, 3> pipe(short_smem, warp, lane, a.status, a.limit_ns);
  const uint32_t qb = static_cast<uint32_t>(Lq) * D * 2, kb = static_cast<uint32_t>(Lk) * D * 2;
  const uint32_t bytes[3] = {qb, kb, kb};
  auto issue = [&](long long seq, int b) {  // Q, K, V
    const void* const src[3] = {q + seq * Lq * D, k + seq * Lk * D, v + seq * Lk * D};
    pipe.issue(b, src, bytes);
  };

  const long long n_warps = static_cast<long long>(gridDim.x) * kShortWarps;
  long long seq = static_cast<long long>(blockIdx.x) * kShortWarps + warp;
  int n = 0;  // this warp's iteration: buffer n % 2, its (n / 2)-th use
  bool ok = true;
  if (seq < a.n_seq && lane == 0) issue(seq, 0);
  for (; seq < a.n_seq; seq += n_warps, ++n) {
    if (seq + n_warps < a.n_seq && lane == 0) issue(seq + n_warps, (n + 1) & 1);
    if (!(ok = pipe.wait(n))) break;
    uint32_t vv[8][D / 32];
    load_cols<D>(vv, pipe.tile(n, 2), Lk, t);
    float sc[2];
    block_scores<D>(pipe.tile(n, 0), pipe.tile(n, 1), Lq, Lk, ga, gb, gs, sc);
    __syncwarp();  // buffer n % 2 is free for the sequence after next

    // softmax of row my_row, base 2
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (my_key + u >= Lk) sc[u] = -INFINITY;
    float m = fmaxf(sc[0], sc[1]);
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
    const float m2 = m * sl2;
    float p[2];
    p[0] = ex2_approx(fmaf(sc[0], sl2, -m2));
    p[1] = ex2_approx(fmaf(sc[1], sl2, -m2));
    float l = p[0] + p[1];
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 8);
    if ((lane & 9) == 0 && my_row < Lq) a.lse[seq * Lq + my_row] = (m2 + lg2_approx(l)) * kLn2;
    const float inv_l = 1.f / l;

    // O = P V / l: the row group's weights, this lane's columns
    float pr[4][8], inv[4];
    gather_rows(pr, p);
#pragma unroll
    for (int r = 0; r < 4; ++r) inv[r] = __shfl_sync(kFull, inv_l, 2 * r, 16);
    product_store<D>(pr, vv, inv, o + (seq * Lq + 4 * ga) * D + t * CW, 4 * ga, Lq);
  }
  if (!ok) pipe.drain(n, seq + n_warps < a.n_seq, lane);
}

template <int D>
__global__ void __launch_bounds__(kShortThreads) bwd_short_kernel(const ShortBwdArgs a) {
  constexpr int CW = D / 16;
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(128) uint8_t short_smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ga = lane >> 4, gb = (lane >> 3) & 1, gs = lane & 7;
  const int t = lane & 15;
  const int Lq = a.Lq, Lk = a.Lk;
  const float sl2 = a.scale_log2;
  const __nv_bfloat16* const q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* const k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* const v = static_cast<const __nv_bfloat16*>(a.v);
  const __nv_bfloat16* const dO = static_cast<const __nv_bfloat16*>(a.dO);
  __nv_bfloat16* const dq = static_cast<__nv_bfloat16*>(a.dq);
  __nv_bfloat16* const dk = static_cast<__nv_bfloat16*>(a.dk);
  __nv_bfloat16* const dv = static_cast<__nv_bfloat16*>(a.dv);
  const int my_row = 4 * ga + (gs >> 1);
  const int my_key = 4 * gb + 2 * (gs & 1);
  const float one[4] = {1.f, 1.f, 1.f, 1.f};
  const float scl[4] = {a.scale, a.scale, a.scale, a.scale};
  ShortPipe<D, 4> pipe(short_smem, warp, lane, a.status, a.limit_ns);
  const uint32_t qb = static_cast<uint32_t>(Lq) * D * 2, kb = static_cast<uint32_t>(Lk) * D * 2;
  const uint32_t bytes[4] = {qb, kb, kb, qb};
  auto issue = [&](long long seq, int b) {  // Q, K, V, dO
    const void* const src[4] = {q + seq * Lq * D, k + seq * Lk * D, v + seq * Lk * D,
                                dO + seq * Lq * D};
    pipe.issue(b, src, bytes);
  };

  const long long n_warps = static_cast<long long>(gridDim.x) * kShortWarps;
  long long seq = static_cast<long long>(blockIdx.x) * kShortWarps + warp;
  int n = 0;
  bool ok = true;
  if (seq < a.n_seq && lane == 0) issue(seq, 0);
  for (; seq < a.n_seq; seq += n_warps, ++n) {
    if (seq + n_warps < a.n_seq && lane == 0) issue(seq + n_warps, (n + 1) & 1);
    const float lse2 = my_row < Lq ? a.lse[seq * Lq + my_row] * kLog2e : 0.f;
    if (!(ok = pipe.wait(n))) break;
    const uint8_t* sq = pipe.tile(n, 0);
    const uint8_t* sk = pipe.tile(n, 1);
    const uint8_t* sv = pipe.tile(n, 2);
    const uint8_t* sdo = pipe.tile(n, 3);
    float sc[2], dp[2];
    block_scores<D>(sq, sk, Lq, Lk, ga, gb, gs, sc);
    block_scores<D>(sdo, sv, Lq, Lk, ga, gb, gs, dp);
    // P, D = sum_j P dP over the row, dS = P (dP - D)
    float p[2], ds[2];
#pragma unroll
    for (int u = 0; u < 2; ++u)
      p[u] = (my_row < Lq && my_key + u < Lk) ? ex2_approx(fmaf(sc[u], sl2, -lse2)) : 0.f;
    float dd = fmaf(p[0], dp[0], p[1] * dp[1]);
    dd += __shfl_xor_sync(kFull, dd, 1);
    dd += __shfl_xor_sync(kFull, dd, 8);
#pragma unroll
    for (int u = 0; u < 2; ++u) ds[u] = p[u] * (dp[u] - dd);

    // dQ = scale dS K: query rows 4a..4a+3
    {
      float w[4][8];
      gather_rows(w, ds);
      uint32_t kc[8][D / 32];
      load_cols<D>(kc, sk, Lk, t);
      product_store<D>(w, kc, scl, dq + (seq * Lq + 4 * ga) * D + t * CW, 4 * ga, Lq);
    }
    // dV = P^T dO and dK = scale dS^T Q: key rows 4a..4a+3
    {
      float w[4][8];
      uint32_t cc[8][D / 32];
      gather_keys(w, p, ga);
      load_cols<D>(cc, sdo, Lq, t);
      product_store<D>(w, cc, one, dv + (seq * Lk + 4 * ga) * D + t * CW, 4 * ga, Lk);
      gather_keys(w, ds, ga);
      load_cols<D>(cc, sq, Lq, t);
      product_store<D>(w, cc, scl, dk + (seq * Lk + 4 * ga) * D + t * CW, 4 * ga, Lk);
    }
    __syncwarp();  // buffer n % 2 is free for the sequence after next
  }
  if (!ok) pipe.drain(n, seq + n_warps < a.n_seq, lane);
}

// One resident wave of persistent blocks, or fewer for few sequences.
template <typename Args>
cudaError_t launch_short_kernel(void (*kern)(Args), int smem_bytes, const Args& a,
                                cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kShortThreads, smem_bytes);
  if (e != cudaSuccess) return e;
  const long long need = (a.n_seq + kShortWarps - 1) / kShortWarps;
  const long long wave = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
  const long long blocks = need < wave ? need : wave;
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kShortThreads), smem_bytes,
                    stream, a);
}

}  // namespace

cudaError_t launch_fwd_short(const ShortArgs& a, int d, cudaStream_t stream) {
  return d == 64 ? launch_short_kernel(fwd_short_kernel<64>, ShortSmem<64, 3>::kBytes, a, stream)
                 : launch_short_kernel(fwd_short_kernel<128>, ShortSmem<128, 3>::kBytes, a, stream);
}

cudaError_t launch_bwd_short(const ShortBwdArgs& a, int d, cudaStream_t stream) {
  return d == 64 ? launch_short_kernel(bwd_short_kernel<64>, ShortSmem<64, 4>::kBytes, a, stream)
                 : launch_short_kernel(bwd_short_kernel<128>, ShortSmem<128, 4>::kBytes, a, stream);
}

}  // namespace eba
