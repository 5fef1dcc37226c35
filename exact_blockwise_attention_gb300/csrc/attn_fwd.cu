// Forward pass of exact blockwise attention on sm_103a (tcgen05 + TMA).
//
// Method: "Training a Large Video Model on a Single Machine in a Day", §3
// "Flash Attention" and §4.1 — attention is computed block by block in on-chip
// memory, with the softmax computed implicitly (online) and block results
// combined without ever storing the Lq x Lk weight matrix. The partial variant
// restricts the keys to [k0, k1) per KV chunk and emits the chunk's own
// normalised output and logsumexp, the unit that split-KV cross-attention
// merges ("LV-XAttn", ICML 2025 poster, Abstract).
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams every
// 128-key tile of its key range past them. Roles:
//   TMA producer warp   Q tiles once, then K_j / V_j into a ring of slots
//   MMA issuer warps    S_t = Q_t K_j^T and O_t += P_t V_j, each issued by a
//                       single elected thread
//   softmax warpgroups  one per query tile, one thread per query row (= TMEM
//                       lane), 128 score columns each
// d = 64: P_t goes back into tensor memory as bf16 and O_t += P_t V_j reads it
//   from there (A operand in TMEM), so P never touches shared memory.
//   TMEM: S_0 [0,128) S_1 [128,256) O_0 [256,320) O_1 [320,384)
//         P_0 [384,448) P_1 [448,512).
//   The QK products and the PV products of each tile are issued by three
//   different threads: one thread issuing N = 64 MMAs with A in tensor memory
//   gets roughly one MMA per ~100 cycles, a third of the tensor pipe, while
//   independent issuing threads add up.
// d = 128: tensor memory is full with S_0, S_1, O_0, O_1, so P_t goes through
//   shared memory as a K-major bf16 operand; one thread issues every MMA.
// No MMA ever reads tensor memory that a later MMA writes.
//
// Online softmax, in base 2 with the scale folded in (x = s * scale * log2 e):
// each row keeps a reference max m and running sums. A tile whose max exceeds
// m by more than 8 (a factor 256) moves m up and rescales O and the sums by
// 2^(m_old - m_new); otherwise the old m is kept, which is exact because O and
// the sums share the same reference. At the end O /= l and lse = (m + log2 l) ln 2.
#include "common.cuh"
#include "kernels.h"

namespace eba {
namespace {

constexpr int kBM = kTileRows;  // query rows per tile
constexpr int kBN = kTileRows;  // keys per tile
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest unrescaled growth
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdCfg {
  static constexpr bool kPTmem = (D == 64);       // P through tensor memory
  static constexpr bool kMultiIssue = (D == 64);  // QK, PV_0, PV_1 from three threads
  static constexpr int kCols = kBN;               // score columns per thread
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kWarpProducer = kSoftmaxWarps;
  static constexpr int kWarpMma = kSoftmaxWarps + 1;  // QK (and PV unless kMultiIssue)
  static constexpr int kThreads = 32 * (kSoftmaxWarps + (kMultiIssue ? 4 : 2));
  static constexpr int kTile = kBM * D * 2;  // bytes of a 128 x D bf16 tile
  static constexpr int kAtom = kBM * 128;    // bytes of one 64-column swizzle atom (16 KB)
  static constexpr int kSlots = (D == 64) ? 8 : 3;
  static constexpr int kP = kPTmem ? 0 : kBM * kBN * 2;
  static constexpr int offQ = 0;
  static constexpr int offKV = offQ + 2 * kTile;
  static constexpr int offP = offKV + kSlots * kTile;
  static constexpr int offBar = offP + 2 * kP;
  // q_full, kv_full[kSlots], kv_empty[kSlots], s_full[2], p_full[2], o_done[2],
  // mma_done[3]
  static constexpr int nBar = 1 + 2 * kSlots + 9;
  static constexpr int offMisc = offBar + nBar * 8;
  static constexpr int kBytes = offMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  // tensor memory columns
  static constexpr uint32_t cS0 = 0, cO0 = 256, cP0 = 384;
  static_assert(!kMultiIssue || kSlots % 2 == 0, "K and V must keep to even / odd slots");
};

template <int D, bool PARTIAL>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FwdArgs args) {
  using L = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x % args.n_pairs;
  const int bh = blockIdx.x / args.n_pairs;
  const int chunk = blockIdx.y;
  const int kbeg = args.bounds[chunk];
  const int kend = args.bounds[chunk + 1];
  const int n_kv = (kend - kbeg + kBN - 1) / kBN;
  const int tile0 = 2 * pair;
  const int n_tiles = min(2, args.n_qtiles - tile0);

  const uint32_t sQ = sbase + L::offQ;
  const uint32_t sKV = sbase + L::offKV;
  const uint32_t sP = sbase + L::offP;
  const uint32_t bar0 = sbase + L::offBar;
  const uint32_t q_full = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (1 + L::kSlots + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (1 + 2 * L::kSlots + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (3 + 2 * L::kSlots + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (5 + 2 * L::kSlots + t); };
  auto mma_done = [&](int i) { return bar0 + 8u * (7 + 2 * L::kSlots + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
  const DeviceStatus st{args.status, args.limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(kv_full(s), 1);
      // With per-tile PV issuers a V slot (odd slots) is released by each tile.
      mbar_init(kv_empty(s), (L::kMultiIssue && (s & 1)) ? n_tiles : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kBM);
      mbar_init(o_done(t), 1);
    }
    for (int i = 0; i < 3; ++i) mbar_init(mma_done(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == L::kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == L::kWarpProducer && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == L::kWarpProducer) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_kv > 0) {
      mbar_arrive_expect_tx(q_full, n_tiles * L::kTile);
      for (int t = 0; t < n_tiles; ++t)
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(sQ + t * L::kTile + a * L::kAtom, &tm_q, q_full, a * 64, (tile0 + t) * kBM,
                      bh);
      int idx = 0;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        for (int w = 0; w < 2; ++w) {
          const int slot = idx % L::kSlots;
          const uint32_t ph = (idx / L::kSlots) & 1;
          if (!mbar_wait(kv_empty(slot), ph ^ 1, abort_flag, st)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(kv_full(slot), L::kTile);
          const CUtensorMap* m = w ? &tm_v : &tm_k;
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(sKV + slot * L::kTile + a * L::kAtom, m, kv_full(slot), a * 64,
                        kbeg + j * kBN, bh);
          ++idx;
        }
      }
      // Every copy started here must land before the CTA may exit.
      mbar_wait_drain(q_full, 0, st);
      for (int i = max(0, idx - L::kSlots); i < idx; ++i)
        mbar_wait_drain(kv_full(i % L::kSlots), (i / L::kSlots) & 1, st);
    }
  } else if (warp >= L::kWarpMma) {
    // ---------------- MMA issuers ----------------
    constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16(kBM, D, false, true);
    // Descriptor words: only the low word (start address >> 4) changes per MMA.
    constexpr uint32_t hi = sdesc_hi(1024);
    const uint32_t q_lo = sdesc_lo(sQ, 16);
    const uint32_t k_lo = sdesc_lo(sKV, 16);
    const uint32_t v_lo = sdesc_lo(sKV, L::kAtom);
    const uint32_t p_lo = sdesc_lo(sP, 16);
    auto slot_off = [&](int idx) { return static_cast<uint32_t>(idx % L::kSlots) * (L::kTile >> 4); };
    // S_t = Q_t K_j^T
    auto issue_qk = [&](int t, int j) {
      const uint32_t a = q_lo + t * (L::kTile >> 4);
      const uint32_t b = k_lo + slot_off(2 * j);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * L::kAtom + (kk & 3) * 32) >> 4;
        mma_ss(tmem + L::cS0 + t * kBN, sdesc_join(a + off, hi), sdesc_join(b + off, hi), idesc_qk,
               kk > 0);
      }
      mma_commit(s_full(t));
    };
    // O_t += P_t V_j (overwrite for j == 0)
    auto issue_pv = [&](int t, int j) {
      const uint32_t b = v_lo + slot_off(2 * j + 1);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint64_t bdesc = sdesc_join(b + kk * (2048 >> 4), hi);
        const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
        if constexpr (L::kPTmem) {
          // 16 keys = 8 columns of packed bf16 per K step
          mma_ts(tmem + L::cO0 + t * D, tmem + L::cP0 + t * 64 + kk * 8, bdesc, idesc_pv, acc);
        } else {
          const uint32_t a = p_lo + ((t * L::kP + (kk >> 2) * L::kAtom + (kk & 3) * 32) >> 4);
          mma_ss(tmem + L::cO0 + t * D, sdesc_join(a, hi), bdesc, idesc_pv, acc);
        }
      }
      mma_commit(o_done(t));
    };
    const int role = warp - L::kWarpMma;  // 0: QK (+PV), 1 / 2: PV of tile 0 / 1
    if (lane == 0 && n_kv > 0 && (role == 0 || role - 1 < n_tiles)) {
      bool ok = true;
      if (role == 0) {
        ok = mbar_wait(q_full, 0, abort_flag, st);
        tc_fence_after();
        // Iteration j issues S_t = Q_t K_j^T (j < n_kv) and, with one issuer,
        // O_t += P_t V_{j-1} (j > 0).
        for (int j = 0; j <= n_kv && ok; ++j) {
          if (L::kMultiIssue && j == n_kv) break;
          if (j < n_kv) {
            if (!mbar_wait(kv_full((2 * j) % L::kSlots), ((2 * j) / L::kSlots) & 1, abort_flag, st))
              break;
            tc_fence_after();
          }
          for (int t = 0; t < n_tiles && ok; ++t) {
            if (j > 0) {
              // softmax of tile t has read S_t and written P_t for KV tile j-1
              if (!mbar_wait(p_full(t), (j - 1) & 1, abort_flag, st)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (j < n_kv) issue_qk(t, j);
            if (!L::kMultiIssue && j > 0) {
              const int iv = 2 * j - 1;
              if (t == 0) {
                if (!mbar_wait(kv_full(iv % L::kSlots), (iv / L::kSlots) & 1, abort_flag, st)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              issue_pv(t, j - 1);
            }
          }
          if (!ok) break;
          if (j < n_kv) mma_commit(kv_empty((2 * j) % L::kSlots));
          if (!L::kMultiIssue && j > 0) mma_commit(kv_empty((2 * j - 1) % L::kSlots));
        }
      } else {
        // PV issuer of tile t: O_t += P_t V_j once the softmax wrote P_t for KV tile j.
        const int t = role - 1;
        for (int j = 0; j < n_kv && ok; ++j) {
          const int iv = 2 * j + 1;
          if (!mbar_wait(p_full(t), j & 1, abort_flag, st) ||
              !mbar_wait(kv_full(iv % L::kSlots), (iv / L::kSlots) & 1, abort_flag, st)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, j);
          mma_commit(kv_empty(iv % L::kSlots));
        }
      }
      // Every MMA this thread issued must be finished before tensor memory is released.
      mma_commit(mma_done(role));
      mbar_wait_drain(mma_done(role), 0, st);
    }
  } else if (warp < L::kSoftmaxWarps) {
    // ---------------- softmax warpgroups ----------------
    const int t = warp >> 2;  // query tile
    const int sub = warp & 3;
    const int r = sub * 32 + lane;  // row within the tile == TMEM lane
    const int row = (tile0 + t) * kBM + r;
    const bool row_ok = row < args.Lq;
    if (t < n_tiles) {
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
      const uint32_t tS = lane_base + L::cS0 + t * kBN;
      const uint32_t tO = lane_base + L::cO0 + t * D;
      const float sl2 = args.scale_log2;
      const float2 sl2v = make_float2(sl2, sl2);
      float m_used = -INFINITY;
      float2 l_sum = make_float2(0.f, 0.f);  // fp32 weights (lse), two lanes
      float2 l_out = make_float2(0.f, 0.f);  // bf16-rounded weights (O normaliser)
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(s_full(t), j & 1, abort_flag, st));
        if (!ok) break;
        tc_fence_after();
        float s[kBN];
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(tS + 0, r0);
          tmem_ld32(tS + 32, r1);
          tmem_ld32(tS + 64, r2);
          tmem_ld32(tS + 96, r3);
          tmem_wait_ld();
          reg_pin(r0);
          reg_pin(r1);
          reg_pin(r2);
          reg_pin(r3);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(r0[i]);
            s[32 + i] = __uint_as_float(r1[i]);
            s[64 + i] = __uint_as_float(r2[i]);
            s[96 + i] = __uint_as_float(r3[i]);
          }
        }
        const int kvalid = kend - (kbeg + j * kBN);
        if (kvalid < kBN) {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (i >= kvalid) s[i] = -INFINITY;
        }
        // Row max: four independent chains of 3-input maxima.
        float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int i = 4; i + 8 <= kBN; i += 8) {
#pragma unroll
          for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], s[i + u], s[i + 4 + u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) m4[u] = fmaxf(m4[u], s[kBN - 4 + u]);
        const float mx2 = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
        const float m_old = m_used;
        const bool bump = mx2 > m_used + kRescaleThreshold;
        if (bump) m_used = mx2;
        // Weights against the reference max, and two row sums: the fp32
        // weights (exact normaliser, for lse) and the bf16-rounded weights that
        // actually multiply V (for O, so O / l is normalised by exactly the
        // weights applied: with a stale reference max the dominant weight is
        // not 1 and its rounding would otherwise scale the whole row).
        const float2 negm = make_float2(-m_used, -m_used);
        uint32_t pk[kBN / 2];
        float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float2 rq[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < kBN / 2; ++i) {
          const float2 x = fma2(make_float2(s[2 * i], s[2 * i + 1]), sl2v, negm);
          const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          pk[i] = pack_bf16(p.x, p.y);
          rs[i & 1] = add2(rs[i & 1], p);
          rq[i & 1] = add2(rq[i & 1], make_float2(bf16lo_f32(pk[i]), bf16hi_f32(pk[i])));
        }
        if (j > 0) {
          // O_t += P_t V_{j-1} must be finished before P_t is overwritten or
          // O_t is rescaled.
          ok = __all_sync(0xffffffffu, mbar_wait(o_done(t), (j - 1) & 1, abort_flag, st));
          if (!ok) break;
          tc_fence_after();
        }
        // P row out first (frees its registers), then the rare O rescale.
        if constexpr (L::kPTmem) {
          // 128 keys = 64 columns of packed bf16 in P_t.
          uint32_t(&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(pk);
          uint32_t(&p1)[32] = *reinterpret_cast<uint32_t(*)[32]>(pk + 32);
          tmem_st32(lane_base + L::cP0 + t * 64, p0);
          tmem_st32(lane_base + L::cP0 + t * 64 + 32, p1);
        } else {
          // P row -> shared memory as a K-major, 128-byte-swizzled bf16 operand:
          // two atoms of 64 keys, 16-byte chunk c of row r at chunk c ^ (r & 7).
          const uint32_t pbase = sP + t * L::kP;
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const int i = a * 32 + ch * 4;
              st_shared_v4(pbase + a * L::kAtom + sw128_offset(r, ch), pk[i], pk[i + 1],
                           pk[i + 2], pk[i + 3]);
            }
          fence_proxy_async_smem();
        }
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          const float alpha = bump ? ex2_approx(m_old - m_used) : 1.f;
          l_sum.x *= alpha;
          l_sum.y *= alpha;
          l_out.x *= alpha;
          l_out.y *= alpha;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + 32 * c, ov);
            tmem_wait_ld();
            reg_pin(ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tO + 32 * c, ov);
          }
        }
        l_sum = add2(l_sum, add2(rs[0], rs[1]));
        l_out = add2(l_out, add2(rq[0], rq[1]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(t));
      }

      // ---------------- epilogue ----------------
      const float ls = l_sum.x + l_sum.y;
      const float lo = l_out.x + l_out.y;
      const size_t orow = static_cast<size_t>(bh) * args.Lq + row;
      float* lse_out = args.lse + static_cast<size_t>(chunk) * args.lse_chunk_stride;
      if (ok && n_kv > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(o_done(t), (n_kv - 1) & 1, abort_flag, st));
        if (ok) {
          tc_fence_after();
          const float inv_l = 1.f / lo;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + 32 * c, ov);
            tmem_wait_ld();
            reg_pin(ov);
            if (row_ok) {
              if (PARTIAL) {
                float4* dst = reinterpret_cast<float4*>(
                    static_cast<float*>(args.o) + static_cast<size_t>(chunk) * args.o_chunk_stride +
                    orow * D + 32 * c);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  dst[v] = make_float4(__uint_as_float(ov[4 * v]) * inv_l,
                                       __uint_as_float(ov[4 * v + 1]) * inv_l,
                                       __uint_as_float(ov[4 * v + 2]) * inv_l,
                                       __uint_as_float(ov[4 * v + 3]) * inv_l);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) +
                                                      orow * D + 32 * c);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const uint32_t* w = ov + 8 * v;
                  dst[v] = make_uint4(
                      pack_bf16(__uint_as_float(w[0]) * inv_l, __uint_as_float(w[1]) * inv_l),
                      pack_bf16(__uint_as_float(w[2]) * inv_l, __uint_as_float(w[3]) * inv_l),
                      pack_bf16(__uint_as_float(w[4]) * inv_l, __uint_as_float(w[5]) * inv_l),
                      pack_bf16(__uint_as_float(w[6]) * inv_l, __uint_as_float(w[7]) * inv_l));
                }
              }
            }
          }
          if (row_ok) lse_out[orow] = (m_used + lg2_approx(ls)) * kLn2;
        }
      } else if (n_kv == 0 && row_ok) {
        // Empty key range: no key contributes.
        if (PARTIAL) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(args.o) +
                                                  static_cast<size_t>(chunk) * args.o_chunk_stride +
                                                  orow * D);
          for (int v = 0; v < D / 4; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        lse_out[orow] = -INFINITY;
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == L::kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool PARTIAL>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdArgs& a, cudaStream_t stream) {
  using L = FwdCfg<D>;
  auto kern = fwd_kernel<D, PARTIAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;

  dim3 grid(static_cast<unsigned>(a.n_pairs) * a.B * a.H, a.n_chunks);
  kern<<<grid, L::kThreads, L::kAlloc, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int d, bool partial, cudaStream_t stream) {
  if (d == 64) return partial ? launch_fwd_t<64, true>(tq, tk, tv, a, stream)
                              : launch_fwd_t<64, false>(tq, tk, tv, a, stream);
  return partial ? launch_fwd_t<128, true>(tq, tk, tv, a, stream)
                 : launch_fwd_t<128, false>(tq, tk, tv, a, stream);
}

}  // namespace eba
