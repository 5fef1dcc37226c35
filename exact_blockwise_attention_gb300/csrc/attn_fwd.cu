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
// Persistent: one CTA per SM walks work items; an item is two 128-row query
// tiles of one (batch, head) (or packed sequence), and every 128-key tile of
// its key range streams past them. Item kinds (template arguments): dense
// [B*H, L, d] heads (query head bh reads K/V head bh / group), packed
// variable-length sequences ([T, H, d]), short sequences packed several to a
// tile (block-diagonal), and an FP8 (e4m3) form of the dense one. Roles:
//   TMA producer warp   Q tiles once, then K_j / V_j into a ring of slots
//   MMA issuer warps    S_t = Q_t K_j^T and O_t += P_t V_j, each issued by a
//                       single elected thread
//   softmax warpgroups  one per query tile, one thread per query row (= TMEM
//                       lane), 128 score columns each
// d = 64: P_t goes back into tensor memory as bf16 and O_t += P_t V_j reads it
//   from there (A operand in TMEM), so P never touches shared memory.
//   TMEM: S_0 [0,128) S_1 [128,256) O_0 [256,320) O_1 [320,384)
//         P_0 [384,448) P_1 [448,512).
// d = 128: tensor memory is full with S_0, S_1, O_0, O_1, so P_t goes through
//   shared memory as a K-major bf16 operand.
// Both: the QK products and the PV products of each tile are issued by three
//   different threads. One thread issuing N = 64 MMAs with A in tensor memory
//   gets roughly one MMA per ~100 cycles, a third of the tensor pipe, while
//   independent issuing threads add up; and with one thread for everything
//   the next round's QK waits in its program order behind both tiles' PV,
//   i.e. behind both softmax warpgroups (at d = 128 that single thread made
//   each round ~2.8x its MMA time).
// No MMA ever reads tensor memory that a later MMA writes.
//
// Online softmax, in base 2 with the scale folded in (x = s * scale * log2 e):
// each row keeps a reference max m and running sums. A tile whose max exceeds
// m by more than 8 (a factor 256) moves m up and rescales O and the sums by
// 2^(m_old - m_new); otherwise the old m is kept, which is exact because O and
// the sums share the same reference. At the end O /= l and lse = (m + log2 l) ln 2.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace eba {
namespace {

constexpr int kBM = kTileRows;  // query rows per tile
constexpr int kBN = kTileRows;  // keys per tile
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest unrescaled growth
constexpr float kLn2 = 0.69314718055994530942f;

// FP8 (d = 128 only): Q, K and V^T are e4m3 (one byte per element), P is
// rounded to e4m3 for the PV product; every operand is K-major, so a 128-row
// tile of 128 one-byte elements is a single 128-byte swizzle atom.
template <int D, bool FP8 = false>
struct FwdCfg {
  static_assert(!FP8 || D == 128, "the FP8 forward is built for d = 128");
  static constexpr int kEsz = FP8 ? 1 : 2;        // bytes per Q/K/V/P element
  static constexpr bool kPTmem = (D == 64);       // P through tensor memory
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kWarpProducer = kSoftmaxWarps;
  // producer, then the issuing threads: QK, PV of tile 0, PV of tile 1
  static constexpr int kWarpMma = kSoftmaxWarps + 1;
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 4);
  static constexpr int kTile = kBM * D * kEsz;  // bytes of a 128 x D tile
  static constexpr int kAtom = kBM * 128;       // bytes of one 128-byte-wide swizzle atom (16 KB)
  static constexpr int kAtoms = D * kEsz / 128;  // atoms per tile row (K extent of Q K^T)
  static constexpr int kAtomCols = 128 / kEsz;   // elements per atom row
  static constexpr int kQBufs = (D == 64 || FP8) ? 2 : 1;  // Q tile pairs in flight across items
  static constexpr int kSlots = FP8 ? 6 : (D == 64) ? 8 : 3;
  static constexpr int kP = kPTmem ? 0 : kBM * kBN * kEsz;
  static constexpr int kPAtoms = kBN * kEsz / 128;  // atoms of a P tile row
  static constexpr int offQ = 0;
  static constexpr int offKV = offQ + kQBufs * 2 * kTile;
  static constexpr int offP = offKV + kSlots * kTile;
  // d = 64: each softmax thread parks its deferred epilogue's m, l, l_fix here
  static constexpr bool kDefer = (D == 64);
  static constexpr int offPend = offP + 2 * kP;
  // and, for packed sequences, the row and head it goes to
  static constexpr int offPendRow = offPend + (kDefer ? 256 * 12 : 0);
  static constexpr int offBar = offPendRow + (kDefer ? 256 * 8 : 0);
  // Packed sequences: ring of item descriptors (64 B each) that the producer
  // fills for the other roles.
  static constexpr int kItemRing = 4;
  static constexpr int kItemBytes = 64;
  // q_full[2], q_empty[2], kv_full[kSlots], kv_empty[kSlots], s_full[2],
  // p_full[2], o_done[2], mma_done[3], s_free[2], exp_turn[2], item_full[R],
  // item_empty[R]
  static constexpr int nBar = 4 + 2 * kSlots + 13 + 2 * kItemRing;
  static constexpr int offMisc = offBar + nBar * 8;
  static constexpr int offItems = (offMisc + 16 + 15) & ~15;
  static constexpr int kBytes = offItems + kItemRing * kItemBytes;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  // tensor memory columns
  static constexpr uint32_t cS0 = 0, cO0 = 256, cP0 = 384;

  // Three full warpgroups: the softmax warpgroups get 200 registers per thread
  // and the producer / MMA warpgroup 104, out of the 168 per thread the launch
  // allocates (384 x 168 = 256 x 200 + 128 x 104). Measured best at d = 64 of
  // 208/88 (the issuers spill), 200/104, 192/120, 184/136 and no split.
  static constexpr uint32_t kRegsSoftmax = 200, kRegsOther = 104, kRegsAtLaunch = 168;
  static_assert(256 * kRegsSoftmax + 128 * kRegsOther == kThreads * kRegsAtLaunch,
                "register split must add up to the launch allocation");
};

// One work item = two query tiles of one (chunk, batch*head), or, for packed
// variable-length sequences, of one (sequence, head). Query tile t's rows
// start at qbeg + qstride * (tile0 + t) and end (exclusive) at qend; round j
// reads the 128 key rows from kbeg + kstride * j, up to kend (rows of the
// [B*H, L, d] view, or tokens of [T, H, d]) of K/V head kvh (query head
// bh / group: consecutive query heads share a K/V head). qstride = kstride =
// 128 except for short sequences packed into tiles.
struct FwdItem {
  int pair, bh, kvh, chunk, kbeg, kend, n_kv, tile0, n_tiles, qbeg, qend, qstride, kstride;
};

__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, const NoVarlen&, int item) {
  FwdItem it;
  const int BH = a.B * a.H;
  it.pair = item % a.n_pairs;
  it.bh = (item / a.n_pairs) % BH;
  it.kvh = it.bh / a.group;  // b * H_kv + h / group, as H = group * H_kv
  it.chunk = item / (a.n_pairs * BH);
  it.kbeg = a.bounds[it.chunk];
  it.kend = a.bounds[it.chunk + 1];
  it.n_kv = (it.kend - it.kbeg + kBN - 1) / kBN;
  it.tile0 = 2 * it.pair;
  it.n_tiles = min(2, a.n_qtiles - it.tile0);
  it.qbeg = 0;
  it.qend = a.Lq;
  it.qstride = kBM;
  it.kstride = kBN;
  return it;
}

// Packed short sequences: tile g holds sequences [g * pack, g * pack + pack)
// (rows from g * pack * Lq of the flattened queries, g * pack * Lk of the
// keys). Item i = tiles 2i and 2i + 1; round j reads tile 2i + j's keys, so
// tile t attends in round t only (in the other round its P is zero).
__device__ __forceinline__ int packed_tiles(const PackedTiles& pt) {
  return (pt.n_seqs + pt.pack - 1) / pt.pack;
}
__device__ __forceinline__ FwdItem fwd_item(const FwdArgs&, const PackedTiles& pt, int item) {
  FwdItem it;
  const int g0 = 2 * item;
  const int s0 = g0 * pt.pack;
  const int ns = min(2 * pt.pack, pt.n_seqs - s0);
  it.pair = item;
  it.bh = 0;
  it.kvh = 0;
  it.chunk = 0;
  it.qbeg = s0 * pt.Lq;
  it.qend = it.qbeg + ns * pt.Lq;
  it.kbeg = s0 * pt.Lk;
  it.kend = it.kbeg + ns * pt.Lk;
  it.qstride = pt.pack * pt.Lq;
  it.kstride = pt.pack * pt.Lk;
  it.tile0 = 0;
  it.n_tiles = min(2, packed_tiles(pt) - g0);
  it.n_kv = it.n_tiles;
  return it;
}

// Items: sequences by decreasing key-tile count, then head, then the
// sequence's query-tile pairs in order (pairs of one sequence are
// consecutive, so CTAs running side by side share its K/V; see VarlenTable).
__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, const VarlenTable& vt, int item) {
  FwdItem it;
  const VarlenPos pos = varlen_pos(vt, a.H, item);
  const int s = pos.seq;
  it.bh = pos.head;  // head
  it.kvh = it.bh / a.group;
  it.pair = pos.idx;
  it.chunk = 0;
  it.kbeg = vt.cu_k[s];
  it.kend = vt.cu_k[s + 1];
  it.n_kv = (it.kend - it.kbeg + kBN - 1) / kBN;
  it.qbeg = vt.cu_q[s];
  it.qend = vt.cu_q[s + 1];
  it.tile0 = 2 * it.pair;
  it.n_tiles = min(2, (it.qend - it.qbeg + kBM - 1) / kBM - it.tile0);
  it.qstride = kBM;
  it.kstride = kBN;
  return it;
}

// Persistent: each CTA walks the work items blockIdx.x, blockIdx.x + gridDim.x,
// ... (consecutive items share K/V, so CTAs running side by side hit in L2).
// Every role walks the same item list; barrier phases run on across items.
//
// VT selects how items map to tiles: NoVarlen (dense [B*H, L, d]), VarlenTable
// (packed variable-length sequences, token-major [T, H, d]; the tensor maps
// view them as (d, H, T), so a tile's coordinates are (column, head, first
// token)) or PackedTiles (short sequences sharing tiles under a
// block-diagonal mask).
//
// FP8: e4m3 Q, K and V^T ([B*H, d, Lk]: the V tile is loaded as 128 d-rows of
// 128 keys, K-major for the PV product), e4m3 P, fp32 accumulation; the
// inputs' dequantisation scales are folded into scale_log2 (Q, K) and o_scale
// (V).
template <int D, bool PARTIAL, typename VT, bool FP8 = false>
__global__ void __launch_bounds__(FwdCfg<D, FP8>::kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FwdArgs args,
               const __grid_constant__ VT vt) {
  constexpr bool VARLEN = std::is_same_v<VT, VarlenTable>;
  constexpr bool PACKED = std::is_same_v<VT, PackedTiles>;
  using L = FwdCfg<D, FP8>;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int n_items;
  if constexpr (VARLEN)
    n_items = vt.total * args.H;
  else if constexpr (PACKED)
    n_items = (packed_tiles(vt) + 1) / 2;
  else
    n_items = args.n_pairs * args.B * args.H * args.n_chunks;
  // 128-row box whose first row is `row` of head `head`.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* m, uint32_t bar, int col, int row, int head) {
    if constexpr (VARLEN)
      tma_load_3d(dst, m, bar, col, head, row);
    else
      tma_load_3d(dst, m, bar, col, row, head);
  };

  const uint32_t sQ = sbase + L::offQ;
  const uint32_t sKV = sbase + L::offKV;
  const uint32_t sP = sbase + L::offP;
  const uint32_t bar0 = sbase + L::offBar;
  auto q_full = [&](int b) { return bar0 + 8u * b; };
  auto q_empty = [&](int b) { return bar0 + 8u * (2 + b); };
  auto kv_full = [&](int s) { return bar0 + 8u * (4 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (4 + L::kSlots + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (4 + 2 * L::kSlots + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (6 + 2 * L::kSlots + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (8 + 2 * L::kSlots + t); };
  auto mma_done = [&](int i) { return bar0 + 8u * (10 + 2 * L::kSlots + i); };
  // s_free(t): the softmax of tile t has loaded S_t into registers, so the next
  // S_t may be computed while it works on this one.
  auto s_free = [&](int t) { return bar0 + 8u * (13 + 2 * L::kSlots + t); };
  // exp_turn(t): the other softmax warpgroup has finished its exponentials of
  // the round, so warpgroup t may start its own (the two take turns).
  auto exp_turn = [&](int t) { return bar0 + 8u * (15 + 2 * L::kSlots + t); };
  // item_full(i): descriptor slot i is written; item_empty(i): every reader
  // has its copy (packed sequences only). Readers: the three MMA issuer
  // threads and the 256 softmax threads.
  auto item_full = [&](int i) { return bar0 + 8u * (17 + 2 * L::kSlots + i); };
  auto item_empty = [&](int i) { return bar0 + 8u * (17 + 2 * L::kSlots + L::kItemRing + i); };
  constexpr int kItemReaders = 3 + 256;
  const uint32_t sItems = sbase + L::offItems;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
  const DeviceStatus st{args.status, args.limit_ns};

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full(b), 1);
      mbar_init(q_empty(b), 1);
    }
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(kv_full(s), 1);
      // With per-tile PV issuers a V slot is released by both tile issuers
      // (one of them only hands it on when its tile is absent) and a K slot
      // by two commits of the QK issuer, so every slot takes two arrivals
      // whatever the ring's length.
      mbar_init(kv_empty(s), 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kBM);
      mbar_init(o_done(t), 1);
      mbar_init(s_free(t), kBM);
      mbar_init(exp_turn(t), kBM);
    }
    for (int i = 0; i < 3; ++i) mbar_init(mma_done(i), 1);
    if constexpr (VARLEN)
      for (int i = 0; i < L::kItemRing; ++i) {
        mbar_init(item_full(i), 1);
        mbar_init(item_empty(i), kItemReaders);
      }
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
  pdl_wait();  // the previous kernel's writes are visible from here on

  // Packed sequences: the producer looks each item up in the sequence table
  // (a binary search over kernel-parameter memory, a chain of dependent
  // loads) and hands it to the other roles through the descriptor ring, so
  // the lookup runs once per item on the thread that works ahead. put_item /
  // get_item: the two sides for item m (running index in this CTA); false
  // when a wait timed out.
  auto put_item = [&](int m, const FwdItem& x) {
    const int slot = m % L::kItemRing;
    if (!mbar_wait(item_empty(slot), ((m / L::kItemRing) & 1) ^ 1, abort_flag, st)) return false;
    const uint32_t p = sItems + L::kItemBytes * slot;
    st_shared_v4(p, x.pair, x.bh, x.kvh, x.chunk);
    st_shared_v4(p + 16, x.kbeg, x.kend, x.n_kv, x.tile0);
    st_shared_v4(p + 32, x.n_tiles, x.qbeg, x.qend, x.qstride);
    st_shared_v4(p + 48, x.kstride, 0u, 0u, 0u);
    mbar_arrive(item_full(slot));
    return true;
  };
  auto get_item = [&](int m, FwdItem& x) {
    const int slot = m % L::kItemRing;
    if (!mbar_wait(item_full(slot), (m / L::kItemRing) & 1, abort_flag, st)) return false;
    const uint32_t p = sItems + L::kItemBytes * slot;
    const uint4 a = ld_shared_v4(p), b = ld_shared_v4(p + 16), c = ld_shared_v4(p + 32);
    const uint4 e = ld_shared_v4(p + 48);
    x.pair = a.x;
    x.bh = a.y;
    x.kvh = a.z;
    x.chunk = a.w;
    x.kbeg = b.x;
    x.kend = b.y;
    x.n_kv = b.z;
    x.tile0 = b.w;
    x.n_tiles = c.x;
    x.qbeg = c.y;
    x.qend = c.z;
    x.qstride = c.w;
    x.kstride = e.x;
    mbar_arrive(item_empty(slot));
    return true;
  };

  if (warp >= L::kWarpProducer) {
   regs_decrease<L::kRegsOther>();
   if (warp == L::kWarpProducer) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int idx = 0;    // K/V loads issued so far (ring position)
      int nq = 0;     // Q tile pairs loaded so far
      bool ok = true;
      int m = 0;  // items handed over (packed sequences)
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const FwdItem it = fwd_item(args, vt, item);
        if (VARLEN && !(ok = put_item(m++, it))) break;
        if (it.n_kv == 0) continue;
        const int qb = nq % L::kQBufs;
        if (!mbar_wait(q_empty(qb), ((nq / L::kQBufs) & 1) ^ 1, abort_flag, st)) break;
        mbar_arrive_expect_tx(q_full(qb), it.n_tiles * L::kTile);
        for (int t = 0; t < it.n_tiles; ++t)
          for (int a = 0; a < L::kAtoms; ++a)
            load_rows(sQ + (qb * 2 + t) * L::kTile + a * L::kAtom, &tm_q, q_full(qb),
                      a * L::kAtomCols, it.qbeg + (it.tile0 + t) * it.qstride, it.bh);
        ++nq;
        for (int j = 0; j < it.n_kv && ok; ++j) {
          for (int w = 0; w < 2; ++w) {
            const int slot = idx % L::kSlots;
            if (!mbar_wait(kv_empty(slot), ((idx / L::kSlots) & 1) ^ 1, abort_flag, st)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(kv_full(slot), L::kTile);
            const CUtensorMap* m = w ? &tm_v : &tm_k;
            if (FP8 && w) {
              // V^T: the d rows of 128 consecutive keys (one atom)
              tma_load_3d(sKV + slot * L::kTile, &tm_v, kv_full(slot), it.kbeg + j * it.kstride, 0,
                          it.kvh);
            } else {
              for (int a = 0; a < L::kAtoms; ++a)
                load_rows(sKV + slot * L::kTile + a * L::kAtom, m, kv_full(slot),
                          a * L::kAtomCols, it.kbeg + j * it.kstride, it.kvh);
            }
            ++idx;
          }
        }
      }
      // Every copy started here must land before the CTA may exit.
      for (int i = max(0, nq - L::kQBufs); i < nq; ++i)
        mbar_wait_drain(q_full(i % L::kQBufs), (i / L::kQBufs) & 1, st);
      for (int i = max(0, idx - L::kSlots); i < idx; ++i)
        mbar_wait_drain(kv_full(i % L::kSlots), (i / L::kSlots) & 1, st);
    }
   } else {
    // ---------------- MMA issuers ----------------
    constexpr uint32_t idesc_qk = FP8 ? idesc_e4m3(kBM, kBN) : idesc_bf16(kBM, kBN, false, false);
    // PV: V is MN-major (bf16), or V^T K-major (FP8)
    constexpr uint32_t idesc_pv = FP8 ? idesc_e4m3(kBM, D) : idesc_bf16(kBM, D, false, true);
    auto mma = [&](uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
      if constexpr (FP8)
        mma_ss_f8(d_tmem, a_desc, b_desc, idesc, acc);
      else
        mma_ss(d_tmem, a_desc, b_desc, idesc, acc);
    };
    // Descriptor words: only the low word (start address >> 4) changes per MMA.
    constexpr uint32_t hi = sdesc_hi(1024);
    const uint32_t q_lo = sdesc_lo(sQ, 16);
    const uint32_t k_lo = sdesc_lo(sKV, 16);
    const uint32_t v_lo = sdesc_lo(sKV, L::kAtom);
    const uint32_t p_lo = sdesc_lo(sP, 16);
    auto slot_off = [&](int idx) { return static_cast<uint32_t>(idx % L::kSlots) * (L::kTile >> 4); };
    // S_t = Q_t K^T with K from ring position kidx
    auto issue_qk = [&](int qb, int t, int kidx) {
      const uint32_t a = q_lo + (qb * 2 + t) * (L::kTile >> 4);
      const uint32_t b = k_lo + slot_off(kidx);
      // K steps of 32 bytes (16 bf16 or 32 e4m3 elements)
#pragma unroll
      for (int kk = 0; kk < D * L::kEsz / 32; ++kk) {
        const uint32_t off = ((kk >> 2) * L::kAtom + (kk & 3) * 32) >> 4;
        mma(tmem + L::cS0 + t * kBN, sdesc_join(a + off, hi), sdesc_join(b + off, hi), idesc_qk,
            kk > 0);
      }
      mma_commit(s_full(t));
    };
    // O_t += P_t V with V from ring position vidx (overwrite when first)
    auto issue_pv = [&](int t, int vidx, bool first) {
      if constexpr (FP8) {
        // A = P_t (e4m3, one atom of 128 keys), B = V^T (d rows of 128 keys):
        // both K-major, K steps of 32 keys
        const uint32_t b = k_lo + slot_off(vidx);
        const uint32_t a = p_lo + ((t * L::kP) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma(tmem + L::cO0 + t * D, sdesc_join(a + kk * 2, hi), sdesc_join(b + kk * 2, hi),
              idesc_pv, (!first || kk > 0) ? 1u : 0u);
        mma_commit(o_done(t));
        return;
      }
      const uint32_t b = v_lo + slot_off(vidx);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint64_t bdesc = sdesc_join(b + kk * (2048 >> 4), hi);
        const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
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
    const int role = warp - L::kWarpMma;  // 0: QK, 1 / 2: PV of tile 0 / 1
    if (lane == 0) {
      bool ok = true;
      int kvbase = 0;         // ring position of this item's K_0
      int nq = 0;             // Q tile pairs consumed
      int uses[2] = {0, 0};   // S_t rounds issued (role 0: s_free phases) or P_t
                              // rounds consumed (PV issuers: p_full phases) per tile
      int m = 0;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++m) {
        FwdItem it;
        if constexpr (VARLEN) {
          if (!(ok = get_item(m, it))) break;
        } else {
          it = fwd_item(args, vt, item);
        }
        if (it.n_kv == 0) continue;
        if (role == 0) {
          const int qb = nq % L::kQBufs;
          if (!(ok = mbar_wait(q_full(qb), (nq / L::kQBufs) & 1, abort_flag, st))) break;
          tc_fence_after();
          // Round j issues S_t = Q_t K_j^T for both tiles.
          for (int j = 0; j < it.n_kv && ok; ++j) {
            const int ik = kvbase + 2 * j;
            if (!(ok = mbar_wait(kv_full(ik % L::kSlots), (ik / L::kSlots) & 1, abort_flag, st)))
              break;
            tc_fence_after();
            for (int t = 0; t < it.n_tiles && ok; ++t) {
              // The softmax of tile t has loaded S_t of its previous round.
              if (uses[t] > 0 && !(ok = mbar_wait(s_free(t), (uses[t] - 1) & 1, abort_flag, st)))
                break;
              tc_fence_after();
              issue_qk(qb, t, ik);
              ++uses[t];
            }
            if (!ok) break;
            // Every ring slot takes two arrivals (a V slot: one per PV issuer);
            // a K slot's are both from this thread.
            mma_commit(kv_empty(ik % L::kSlots));
            mma_commit(kv_empty(ik % L::kSlots));
          }
          // Q tiles free once this item's QK products are done.
          mma_commit(q_empty(qb));
          ++nq;
        } else {
          // PV issuer of tile t: O_t += P_t V_j once the softmax wrote P_t for
          // KV tile j. When the item has no tile t, only hand the V slots on.
          const int t = role - 1;
          for (int j = 0; j < it.n_kv && ok; ++j) {
            const int iv = kvbase + 2 * j + 1;
            if (t < it.n_tiles) {
              if (!(ok = mbar_wait(p_full(t), uses[t] & 1, abort_flag, st))) break;
              ++uses[t];
            }
            if (!(ok = mbar_wait(kv_full(iv % L::kSlots), (iv / L::kSlots) & 1, abort_flag, st)))
              break;
            if (t < it.n_tiles) {
              tc_fence_after();
              issue_pv(t, iv, j == 0);
              mma_commit(kv_empty(iv % L::kSlots));
            } else {
              mbar_arrive(kv_empty(iv % L::kSlots));
            }
          }
        }
        kvbase += 2 * it.n_kv;
      }
      // Every MMA this thread issued must be finished before tensor memory is released.
      mma_commit(mma_done(role));
      mbar_wait_drain(mma_done(role), 0, st);
    }
   }
  } else {
    regs_increase<L::kRegsSoftmax>();
    // ---------------- softmax warpgroups ----------------
    const int t = warp >> 2;  // query tile of the item
    const int sub = warp & 3;
    const int r = sub * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const uint32_t tS = lane_base + L::cS0 + t * kBN;
    const uint32_t tO = lane_base + L::cO0 + t * D;
    const float sl2 = args.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    bool ok = true;
    int rounds = 0;  // S_t / P_t / O_t rounds of this tile so far (barrier phases)
    // The two warpgroups take turns on the exponentials (the MUFU pipe is
    // shared): warpgroup 0 goes first in every round. turns counts the rounds
    // of every item, including those of items without this warpgroup's tile.
    int turns = 0;
    auto wait_turn = [&]() {
      return __all_sync(0xffffffffu, mbar_wait(exp_turn(t), t == 0 ? ((turns & 1) ^ 1) : (turns & 1),
                                                abort_flag, st));
    };
    auto pass_turn = [&]() {
      mbar_arrive(exp_turn(1 - t));
      ++turns;
    };
    // d = 64: an item's epilogue (O / l out of tensor memory, then to HBM,
    // and lse) is deferred into this warpgroup's next round 0: there O_t is
    // read after the new P_t is stored and before p_full lets the PV that
    // overwrites O_t start, so the item's last P V runs under the next
    // item's first softmax. Only the item index stays in a register; m, l
    // and l_fix wait in shared memory, the row's offsets are recomputed.
    float* pend_f = reinterpret_cast<float*>(smem + L::offPend) + 3 * threadIdx.x;
    // packed sequences: the pending row (-1: none) and its head, as the item's
    // descriptor is gone from the ring by then
    int2* pend_row = reinterpret_cast<int2*>(smem + L::offPendRow) + threadIdx.x;
    int pend_item = -1;
    auto store_pending = [&](const uint32_t* ov) {
      int prow, pbh, pchunk;
      bool prow_ok;
      if constexpr (VARLEN) {
        const int2 pr = *pend_row;
        prow = pr.x;
        pbh = pr.y;
        pchunk = 0;
        prow_ok = prow >= 0;
      } else {
        const FwdItem pit = fwd_item(args, vt, pend_item);
        prow = pit.qbeg + (pit.tile0 + t) * pit.qstride + r;
        pbh = pit.bh;
        pchunk = pit.chunk;
        prow_ok = prow < pit.qend;
        if constexpr (PACKED) {
          const int ns = min(vt.pack, vt.n_seqs - (2 * pend_item + t) * vt.pack);
          prow_ok = r < ns * vt.Lq;
        }
      }
      pend_item = -1;
      if (!prow_ok) return;
      const size_t porow = static_cast<size_t>(pbh) * args.Lq + prow;
      const size_t po_off = VARLEN ? (static_cast<size_t>(prow) * args.H + pbh) * D : porow * D;
      const float pm = pend_f[0], pls = pend_f[1], plo = pend_f[2];
      const float inv_l = 1.f / plo;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        const uint32_t* oc = ov + 32 * c;
        if (PARTIAL) {
          float4* dst = reinterpret_cast<float4*>(
              static_cast<float*>(args.o) + static_cast<size_t>(pchunk) * args.o_chunk_stride +
              porow * D + 32 * c);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(oc[4 * v]) * inv_l, __uint_as_float(oc[4 * v + 1]) * inv_l,
                                 __uint_as_float(oc[4 * v + 2]) * inv_l,
                                 __uint_as_float(oc[4 * v + 3]) * inv_l);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) + po_off + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t* w = oc + 8 * v;
            dst[v] = make_uint4(
                pack_bf16(__uint_as_float(w[0]) * inv_l, __uint_as_float(w[1]) * inv_l),
                pack_bf16(__uint_as_float(w[2]) * inv_l, __uint_as_float(w[3]) * inv_l),
                pack_bf16(__uint_as_float(w[4]) * inv_l, __uint_as_float(w[5]) * inv_l),
                pack_bf16(__uint_as_float(w[6]) * inv_l, __uint_as_float(w[7]) * inv_l));
          }
        }
      }
      float* lse_p = args.lse + static_cast<size_t>(pchunk) * args.lse_chunk_stride;
      lse_p[porow] = (pm + lg2_approx(pls)) * kLn2;
    };
    auto read_o = [&](uint32_t (&ov)[D]) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(ov + 32 * c));
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) reg_pin(*reinterpret_cast<uint32_t(*)[32]>(ov + 32 * c));
    };
    // The pending epilogue on its own (no round of this tile follows).
    auto flush = [&]() -> bool {
      if (pend_item < 0) return true;
      if (!__all_sync(0xffffffffu, mbar_wait(o_done(t), (rounds - 1) & 1, abort_flag, st))) return false;
      tc_fence_after();
      uint32_t ov[D];
      read_o(ov);
      tc_fence_before();
      store_pending(ov);
      return true;
    };
    int m = 0;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++m) {
      FwdItem it;
      if constexpr (VARLEN) {
        if (!(ok = __all_sync(0xffffffffu, get_item(m, it)))) break;
      } else {
        it = fwd_item(args, vt, item);
      }
      if (t >= it.n_tiles) {
        if (!(ok = flush())) break;
        // No tile for this warpgroup: only keep the turns going.
        for (int j = 0; j < it.n_kv && ok; ++j) {
          if (!(ok = wait_turn())) break;
          pass_turn();
        }
        continue;
      }
      const int row = it.qbeg + (it.tile0 + t) * it.qstride + r;
      bool row_ok = row < it.qend;
      if constexpr (PACKED) {
        // this tile's sequences only (the next tile's rows follow it directly)
        const int ns = min(vt.pack, vt.n_seqs - (2 * item + t) * vt.pack);
        row_ok = r < ns * vt.Lq;
      }
      const size_t orow = static_cast<size_t>(it.bh) * args.Lq + row;  // lse index ([H, T] when packed)
      // element offset of this row of O: [B*H, Lq, d], or token-major [T, H, d]
      const size_t o_off = VARLEN ? (static_cast<size_t>(row) * args.H + it.bh) * D : orow * D;
      float* lse_out = args.lse + static_cast<size_t>(it.chunk) * args.lse_chunk_stride;
      if (it.n_kv == 0) {
        if (!(ok = flush())) break;
        // Empty key range: no key contributes.
        if (row_ok) {
          if (PARTIAL) {
            float4* dst = reinterpret_cast<float4*>(
                static_cast<float*>(args.o) + static_cast<size_t>(it.chunk) * args.o_chunk_stride +
                orow * D);
            for (int v = 0; v < D / 4; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else if (VARLEN) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) + o_off);
            for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
          }
          lse_out[orow] = -INFINITY;
        }
        continue;
      }
      float m_used = -INFINITY;
      float2 l_sum = make_float2(0.f, 0.f);  // sum of the fp32 weights (lse), two lanes
      float l_fix = 0.f;  // rounding error of each tile's largest bf16 weight (O normaliser)
      for (int j = 0; j < it.n_kv; ++j, ++rounds) {
        ok = __all_sync(0xffffffffu, mbar_wait(s_full(t), rounds & 1, abort_flag, st));
        if (!ok) break;
        tc_fence_after();
        if (PACKED && j != t) {
          // Packed tiles: round j holds the other tile's keys. P_t = 0, so
          // O_t, the row max and the row sum are unchanged; the barriers and
          // turns run as in any round.
          tc_fence_before();
          mbar_arrive(s_free(t));
          if (!(ok = wait_turn())) break;
          pass_turn();
          if (j > 0 || pend_item >= 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(o_done(t), (rounds - 1) & 1, abort_flag, st));
            if (!ok) break;
            tc_fence_after();
          }
          if constexpr (L::kPTmem) {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            tmem_st32(lane_base + L::cP0 + t * 64, z);
            tmem_st32(lane_base + L::cP0 + t * 64 + 32, z);
            tmem_st_wait();
          } else {
            const uint32_t pbase = sP + t * L::kP;
#pragma unroll
            for (int a = 0; a < L::kPAtoms; ++a)
#pragma unroll
              for (int ch = 0; ch < 8; ++ch)
                st_shared_v4(pbase + a * L::kAtom + sw128_offset(r, ch), 0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
          }
          if (L::kDefer && pend_item >= 0) {
            uint32_t ov[D];
            read_o(ov);
            tc_fence_before();
            mbar_arrive(p_full(t));
            store_pending(ov);
            continue;
          }
          tc_fence_before();
          mbar_arrive(p_full(t));
          continue;
        }
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
          tc_fence_before();
          mbar_arrive(s_free(t));  // S_t may be overwritten by the next round's QK
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(r0[i]);
            s[32 + i] = __uint_as_float(r1[i]);
            s[64 + i] = __uint_as_float(r2[i]);
            s[96 + i] = __uint_as_float(r3[i]);
          }
        }
        const int kvalid = it.kend - (it.kbeg + j * kBN);
        if (!PACKED && kvalid < kBN) {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (i >= kvalid) s[i] = -INFINITY;
        }
        if constexpr (PACKED) {
          // Block-diagonal: the row's own sequence's keys only. (Rows past the
          // tile's sequences see no key; they are never stored.)
          const int lo = (r / vt.Lq) * vt.Lk, hi = lo + vt.Lk;
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (i < lo || i >= hi) s[i] = -INFINITY;
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
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float mx2 = mx * sl2;
        const float m_old = m_used;
        const bool bump = mx2 > m_used + kRescaleThreshold;
        if (bump) m_used = mx2;
        // Weights against the reference max and their fp32 row sum (the exact
        // normaliser, for lse). O is normalised by the sum of the bf16-rounded
        // weights that actually multiply V: with a stale reference max the
        // tile's largest weight is not 1, and its rounding alone would scale
        // the whole row. That sum is the fp32 sum plus the rounding errors;
        // only the largest weight's error matters at this precision, so only
        // it is added (l_fix), at one exponential per row and tile.
        const float2 negm = make_float2(-m_used, -m_used);
        if (!(ok = wait_turn())) break;
        // P row packed for the PV product: bf16 pairs, or (FP8) e4m3 quads
        uint32_t pk[kBN * L::kEsz / 4];
        float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if constexpr (FP8) {
#pragma unroll
          for (int i = 0; i < kBN / 4; ++i) {
            const float2 x0 = fma2(make_float2(s[4 * i], s[4 * i + 1]), sl2v, negm);
            const float2 x1 = fma2(make_float2(s[4 * i + 2], s[4 * i + 3]), sl2v, negm);
            const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
            const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
            pk[i] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
            rs[0] = add2(rs[0], p0);
            rs[1] = add2(rs[1], p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kBN / 2; ++i) {
            const float2 x = fma2(make_float2(s[2 * i], s[2 * i + 1]), sl2v, negm);
            const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            pk[i] = pack_bf16(p.x, p.y);
            rs[i & 1] = add2(rs[i & 1], p);
          }
        }
        const float pmax = ex2_approx(fmaf(mx, sl2, -m_used));
        const float pmax_err =
            (FP8 ? round_e4m3(pmax) : bf16lo_f32(pack_bf16(pmax, 0.f))) - pmax;
        pass_turn();
        if (j > 0 || pend_item >= 0) {
          // O_t += P_t V_{j-1} (or the previous item's last P V) must be
          // finished before P_t is overwritten or O_t is rescaled or read.
          ok = __all_sync(0xffffffffu, mbar_wait(o_done(t), (rounds - 1) & 1, abort_flag, st));
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
          // P row -> shared memory as a K-major, 128-byte-swizzled operand:
          // atoms of 128 bytes (64 bf16 or 128 e4m3 keys), 16-byte chunk c of
          // row r at chunk c ^ (r & 7).
          const uint32_t pbase = sP + t * L::kP;
#pragma unroll
          for (int a = 0; a < L::kPAtoms; ++a)
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
          l_fix *= alpha;
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
        l_fix += pmax_err;
        tmem_st_wait();
        if (L::kDefer && pend_item >= 0) {
          // the previous item's O_t, read before this round's PV overwrites it
          uint32_t ov[D];
          read_o(ov);
          tc_fence_before();
          mbar_arrive(p_full(t));
          store_pending(ov);
          continue;
        }
        tc_fence_before();
        mbar_arrive(p_full(t));
      }
      if (!ok) break;

      // ---------------- epilogue of the item ----------------
      const float ls = l_sum.x + l_sum.y;
      const float lo = ls + l_fix;
      if constexpr (L::kDefer) {
        pend_f[0] = m_used;
        pend_f[1] = ls;
        pend_f[2] = lo;
        if constexpr (VARLEN) *pend_row = make_int2(row_ok ? row : -1, it.bh);
        pend_item = item;
        continue;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(o_done(t), (rounds - 1) & 1, abort_flag, st));
      if (!ok) break;
      tc_fence_after();
      const float inv_l = (FP8 ? args.o_scale : 1.f) / lo;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + 32 * c, ov);
        tmem_wait_ld();
        reg_pin(ov);
        if (row_ok) {
          if (PARTIAL) {
            float4* dst = reinterpret_cast<float4*>(
                static_cast<float*>(args.o) + static_cast<size_t>(it.chunk) * args.o_chunk_stride +
                orow * D + 32 * c);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(ov[4 * v]) * inv_l,
                                   __uint_as_float(ov[4 * v + 1]) * inv_l,
                                   __uint_as_float(ov[4 * v + 2]) * inv_l,
                                   __uint_as_float(ov[4 * v + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) + o_off +
                                                  32 * c);
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
      // The next item's first P_t V overwrites O_t only after this warpgroup
      // arrives on p_full again, i.e. after these loads.
      tc_fence_before();
    }
    if (ok) ok = flush();
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

template <int D, bool PARTIAL, typename VT, bool FP8 = false>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdArgs& a, const VT& vt, long long items, cudaStream_t stream) {
  using L = FwdCfg<D, FP8>;
  auto kern = fwd_kernel<D, PARTIAL, VT, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  {
    // The warpgroups' register shares must fit the launch allocation, or an
    // increase would wait forever: refuse to launch otherwise.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < static_cast<int>(L::kRegsAtLaunch)) return cudaErrorInvalidConfiguration;
  }

  // Persistent grid: one CTA per SM (tensor memory allows no more), never
  // more CTAs than work items.
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  if (grid == 0) return cudaSuccess;
  return launch_pdl(kern, dim3(grid), dim3(L::kThreads), L::kAlloc, stream, tq, tk, tv, a, vt);
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int d, bool partial, cudaStream_t stream) {
  const long long items = static_cast<long long>(a.n_pairs) * a.B * a.H * a.n_chunks;
  const NoVarlen nv{};
  if (d == 64) return partial ? launch_fwd_t<64, true>(tq, tk, tv, a, nv, items, stream)
                              : launch_fwd_t<64, false>(tq, tk, tv, a, nv, items, stream);
  return partial ? launch_fwd_t<128, true>(tq, tk, tv, a, nv, items, stream)
                 : launch_fwd_t<128, false>(tq, tk, tv, a, nv, items, stream);
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const FwdArgs& a, cudaStream_t stream) {
  const long long items = static_cast<long long>(a.n_pairs) * a.B * a.H;
  return launch_fwd_t<128, false, NoVarlen, true>(tq, tk, tvt, a, NoVarlen{}, items, stream);
}

cudaError_t launch_fwd_packed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdArgs& a, const PackedTiles& pt, int d, cudaStream_t stream) {
  const long long tiles = (static_cast<long long>(pt.n_seqs) + pt.pack - 1) / pt.pack;
  const long long items = (tiles + 1) / 2;  // two tiles per item
  return d == 64 ? launch_fwd_t<64, false>(tq, tk, tv, a, pt, items, stream)
                 : launch_fwd_t<128, false>(tq, tk, tv, a, pt, items, stream);
}

cudaError_t launch_fwd_varlen(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdArgs& a, const VarlenTable& vt, int d, cudaStream_t stream) {
  const long long items = static_cast<long long>(vt.total) * a.H;
  return d == 64 ? launch_fwd_t<64, false>(tq, tk, tv, a, vt, items, stream)
                 : launch_fwd_t<128, false>(tq, tk, tv, a, vt, items, stream);
}

}  // namespace eba
