// Backward pass of exact blockwise attention on sm_103a (tcgen05 + TMA).
//
// Only O and lse are kept from the forward pass; P is recomputed tile by tile
// from lse (activation recomputation, "LV-XAttn", ICML 2025 poster, Abstract;
// the blockwise method of "Training a Large Video Model on a Single Machine in
// a Day", §3/§4.1, is what makes this recomputation cheap in memory). With
// D_i = sum_k dO_ik O_ik (equal to sum_j P_ij dP_ij, the row term of the
// softmax Jacobian):
//   P = exp(S - lse),  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dK = scale * dS^T Q,  dQ = scale * dS K.
//
// Three kernels on one stream:
//   bwd_pre_kernel   D_i and lse_i * log2(e) per row (padded to 128-row tiles),
//                    and zeroes the fp32 dQ accumulator
//   bwd_kernel       persistent (one CTA per SM); a work item is one 128-key
//                    tile against all 128-row query tiles that attend to it;
//                    dK, dV accumulate in tensor memory, dQ tiles are added
//                    into the fp32 accumulator atomically
//   bwd_dq_kernel    dQ = bf16(scale * accumulator)
// Work items come in four kinds (template arguments): dense [B*H, L, d]
// heads; grouped-query heads (an item walks the query tiles of every head of
// its group); packed variable-length sequences ([T, H, d], per-sequence
// bounds); short sequences packed several to a tile (block-diagonal; each
// query row gets all of its dQ from one tile, so dQ is stored directly and
// the accumulator, its zeroing and bwd_dq_kernel are skipped).
//
// bwd_kernel roles (512 threads):
//   warps 0-7    two "compute" warpgroups; warpgroup w handles query columns
//                [64w, 64w+64) of S^T / dP^T for every key row (TMEM lane)
//   warps 8-11   dQ warpgroup: reads dQ tiles out of TMEM, stages them in
//                shared memory and adds them into the fp32 accumulator by
//                TMA reduce-add, whole 128-byte lines (d = 64: own staging
//                buffer; d = 128: the tile's finished Q/dO stage slot)
//   warp 12      issues S^T = K Q^T and dP^T = V dO^T
//   warp 13      issues dV += P^T dO (once P^T is written) and then, once
//                dS^T is written, dQ = dS K
//   warp 14      TMA producer (K, V once; Q_i, dO_i, -lse2_i, D_i per stage)
//   warp 15      issues dK += dS^T Q
// dK and dQ both wait for dS^T and, together, release it (and the next dS^T
// store): issuing them from two threads halves that wait.
// Every accumulator has exactly one issuing thread (so its MMAs stay in one
// in-order stream). Several issuing threads are needed because one thread
// gets only about one N = 64 MMA per ~110 cycles, a third of the tensor pipe.
// Roles that wait on different barriers sit in different warps: a lane that
// is suspended in an mbarrier wait holds up the other lanes of its warp.
// Tensor memory (512 columns):
//   d = 64 : S^T [0,128) dP^T [128,256) dV [256,320) dK [320,384) dQ [384,448)
//            P^T [448,512) as packed bf16, the A operand of dV
//   d = 128: S^T [0,128) dP^T/dQ [128,256) dV [256,384) dK [384,512); P^T
//            reuses S^T: warpgroup w's half at [64w, 64w+32)
// dS^T always goes through shared memory: it is the K-major A of dK and, read
// MN-major, the A of dQ.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace eba {
namespace {

constexpr int kBM = kTileRows;  // keys per KV tile (MMA M)
constexpr int kBN = kTileRows;  // queries per Q tile
constexpr int kThreads = 512;
constexpr int kWarpDq = 8;
constexpr int kWarpIssue = 12;  // first warp of the producer / MMA-issuer warpgroup
constexpr int kWarpSdp = 12;    // S^T and dP^T issuer
constexpr int kWarpDvDq = 13;   // dV and dQ issuer
constexpr int kWarpLoad = 14;   // TMA producer; allocates tensor memory
constexpr int kWarpDk = 15;     // dK issuer
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
// Register split between the four warpgroups (launched with 128 per thread):
// compute warpgroups 168, dQ warpgroup 104, producer / MMA-issuer warpgroup 72.
constexpr uint32_t kRegsCompute = 168, kRegsDq = 104, kRegsIssue = 72;
constexpr int kRegsAtLaunch = (256 * kRegsCompute + 128 * kRegsDq + 128 * kRegsIssue) / kThreads;
static_assert(kRegsAtLaunch == 128, "register split must add up to the launch allocation");

template <int D, int KB>
struct BwdSmem {
  static constexpr bool kDqAlias = (D == 128);  // dQ reuses the dP^T columns
  // P^T (bf16) is the tensor-memory A operand of dV. d = 64: in columns of its
  // own. d = 128: tensor memory is full, so each compute warpgroup writes its
  // half of P^T into the first 32 of its own 64 S^T columns once it has read
  // them (the next S^T then also waits for dV).
  static constexpr bool kPAlias = (D == 128);
  // dQ tiles are added into the fp32 accumulator by TMA reduce-add from a
  // shared-memory staging copy: d = 64 in a buffer of its own; d = 128 (no
  // room for 64 KB more) in the tile's own Q/dO stage slot, once dK, dQ and
  // dV of the tile are done with it.
  static constexpr bool kDqInStage = (D == 128);
  // Where an item's dK, dV leave tensor memory: d = 64 on the dQ warpgroup, so
  // the compute warps start the next item's first tile at once; d = 128 (64 KB
  // of dK, dV per item, and the dQ warpgroup already staging 64 KB dQ tiles)
  // on the compute warps, which measured faster there.
  static constexpr bool kEpiOnDq = (D == 64);
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr int kTile = kBM * D * 2;
  static constexpr int kAtom = kBM * 128;  // 16 KB
  static constexpr int kVec = kBN * 4;     // 512 B: one fp32 value per query row
  static constexpr int kStage = 2 * kTile + 2 * kVec;  // Q_i, dO_i, -lse2_i, D_i
  // K buffers: with two (d = 64, chosen for dense heads with items of at most
  // 32 query tiles), the next item's K loads while this item's last tiles
  // still read K, which shortens item boundaries; long items run faster with
  // one (measured: 196 / 392 / 1568-token heads −5.4 / −3.0 / −0.4 %,
  // 12544-token +1.6 %). Packed sequences always take one (see launch_bwd_k).
  static constexpr int kKBufs = KB;
  static_assert(KB == 1 || (KB == 2 && D == 64), "a second K buffer fits at d = 64 only");
  static constexpr int offK = 0;
  static constexpr int offV = offK + kKBufs * kTile;
  static constexpr int offStage = offV + kTile;
  static constexpr int offDS = offStage + kStages * kStage;  // dS^T bf16
  static constexpr int kDsBytes = kBM * kBN * 2;
  static constexpr int offDQ = offDS + kDsBytes;  // fp32 dQ staging (TMA reduce)
  static constexpr int offBar = offDQ + (kDqInStage ? 0 : kBN * D * 4);
  // Packed sequences: ring of item descriptors (48 B each) that the producer
  // fills for the other roles.
  static constexpr int kItemRing = 4;
  static constexpr int kItemBytes = 48;
  // k_full[KB], k_empty[KB], v_full, v_empty, st_full[S], st_empty[S],
  // dv_slot[S], 16 single barriers, then item_full[R], item_empty[R]
  static constexpr int nBar = 2 * kKBufs + 2 + 3 * kStages + 16 + 2 * kItemRing;
  static constexpr int offMisc = offBar + nBar * 8;
  static constexpr int offItems = (offMisc + 16 + 15) & ~15;
  static constexpr int kBytes = offItems + kItemRing * kItemBytes;
  // d = 128 fills shared memory to within a few hundred bytes of the limit,
  // leaving no room to realign the base: the kernel checks instead that the
  // dynamic shared memory starts on a 1024-byte boundary.
  static constexpr bool kAlignSlack = (D == 64);
  static constexpr int kAlloc = kBytes + (kAlignSlack ? 1024 : 0);
  // TMEM columns
  static constexpr uint32_t cS = 0, cDP = 128, cDV = 256, cDK = 256 + D;
  static constexpr uint32_t cDQ = kDqAlias ? 128 : 256 + 2 * D;
  static constexpr uint32_t cP = kPAlias ? cS : 448;
  // Column where compute warpgroup wg stores its 64 queries of P^T, and the
  // column of dV's K step kk (16 queries = 8 packed columns).
  static __device__ __forceinline__ uint32_t p_store_col(int wg) {
    return kPAlias ? cS + 64 * wg : cP + 32 * wg;
  }
  static __device__ __forceinline__ uint32_t p_col(int kk) {
    return kPAlias ? cS + kk * 8 + (kk >= 4 ? 32 : 0) : cP + kk * 8;
  }
  static_assert(kStage % 1024 == 0 || kStages == 1, "stages must stay 1024-byte aligned");
  static_assert(kBytes + (kAlignSlack ? 1024 : 0) <= 232448, "shared memory over the limit");
};

// One work item: a 128-key tile of one (batch, K/V head), or, for packed
// variable-length sequences, of one (sequence, K/V head), against the nq1
// query tiles of the same sequence of every query head that reads this K/V
// head (group of them, consecutive: nq = group * nq1 tiles). Keys are rows
// [kbeg + 128 ktile, ...) up to kend (exclusive) of K/V head kvh; the item's
// tile i is tile i % nq1 of query head qh0 + i / nq1 (see QCursor).
struct BwdItem {
  int kvh, qh0, ktile, nq1, nq, kbeg, kend, qbeg;
  size_t vbase;  // -lse2 / D offset of query head qh0's first tile
};

__device__ __forceinline__ BwdItem bwd_item(const BwdArgs& a, const NoVarlen&, int w) {
  BwdItem it;
  it.ktile = w % a.n_ktiles;
  it.kvh = w / a.n_ktiles;        // b * H_kv + K/V head
  it.qh0 = it.kvh * a.group;      // b * H + first query head of the group
  it.nq1 = a.n_qtiles;
  it.nq = a.group * it.nq1;
  it.kbeg = 0;
  it.kend = a.Lk;
  it.qbeg = 0;
  it.vbase = static_cast<size_t>(it.qh0) * a.Lq_pad;
  return it;
}

// Walks an item's tiles in order: tile i is tile ti = i % nq1 of query head
// qh0 + gq, gq = i / nq1 (kept as counters, no division). Without grouped
// query heads nq1 = nq, so gq stays 0.
template <bool GQA>
struct QCursor {
  int gq = 0, ti = 0;
  __device__ __forceinline__ int head(const BwdItem& it) const { return it.qh0 + gq; }
  __device__ __forceinline__ int row(const BwdItem& it) const { return it.qbeg + ti * kBN; }
  // -lse2 / D offset of the tile (lq_pad: rows per query head)
  __device__ __forceinline__ size_t voff(const BwdItem& it, int lq_pad) const {
    return it.vbase + static_cast<size_t>(gq) * lq_pad + static_cast<size_t>(ti) * kBN;
  }
  __device__ __forceinline__ void next(const BwdItem& it) {
    ++ti;
    if (GQA && ti == it.nq1) {
      ti = 0;
      ++gq;
    }
  }
};

// Sequence s with cu[s] <= p < cu[s + 1] (cu non-decreasing, cu[0] = 0 <= p <
// cu[n]); empty sequences are skipped.
__device__ __forceinline__ int seq_of(const int* cu, int n, int p) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= p) lo = mid; else hi = mid;
  }
  return lo;
}

// Item w: tile w of packed short sequences, the one key tile against the one
// query tile holding the same sequences; -lse2 / D of tile w at [128 w, 128 w + 128).
__device__ __forceinline__ BwdItem bwd_item(const BwdArgs&, const PackedTiles& pt, int w) {
  BwdItem it;
  const int s0 = w * pt.pack;
  const int ns = min(pt.pack, pt.n_seqs - s0);
  it.kvh = 0;
  it.qh0 = 0;
  it.ktile = 0;
  it.nq1 = 1;
  it.nq = 1;
  it.kbeg = s0 * pt.Lk;
  it.kend = it.kbeg + ns * pt.Lk;
  it.qbeg = s0 * pt.Lq;
  it.vbase = static_cast<size_t>(w) * kBN;
  return it;
}

// Items: sequences by decreasing query-tile count, then K/V head, then the
// sequence's key tiles in order (see VarlenTable).
__device__ __forceinline__ BwdItem bwd_item(const BwdArgs& a, const VarlenTable& vt, int w) {
  BwdItem it;
  const VarlenPos pos = varlen_pos(vt, a.H_kv, w);
  const int s = pos.seq;
  it.kvh = pos.head;  // K/V head
  it.qh0 = it.kvh * a.group;
  it.ktile = pos.idx;
  it.nq1 = vt.cu_qt[s + 1] - vt.cu_qt[s];
  it.nq = a.group * it.nq1;
  it.kbeg = vt.cu_k[s];
  it.kend = vt.cu_k[s + 1];
  it.qbeg = vt.cu_q[s];
  it.vbase = static_cast<size_t>(it.qh0) * a.Lq_pad + static_cast<size_t>(vt.cu_qt[s]) * kBN;
  return it;
}

// Persistent: CTA c takes work items c, c + gridDim.x, ...; consecutive items
// are key tiles of one head (and sequence), sharing its Q and dO tiles, so CTAs
// running side by side hit in L2. Every role walks the same items; barrier
// phases run on across items, counted by the CTA's running query-tile index
// g = (tiles of its earlier items) + i and its running item index n.
//
// VT = VarlenTable: packed sequences, token-major [T, H, d]; the tensor maps
// view them as (d, H, T), so a tile's coordinates are (column, head, first
// token). Query rows of a tile past its sequence's end belong to the next
// sequence: their -lse2 (padding, -inf) makes their P exactly 0, so they add
// nothing to dK, dV and exactly 0 to those rows of dQ. A sequence without
// queries has no items (the host zeroes its dK, dV rows). The producer looks
// every item up in the table and passes it to the other roles through a ring
// of descriptors in shared memory: the lookup (a binary search over
// kernel-parameter memory, a chain of dependent loads) then runs once per
// item, on one thread that works ahead, and not on every role at every item
// start.
// VT = PackedTiles: short sequences sharing tiles; P is kept to the
// block-diagonal (a key row's own sequence's queries), so the other
// sequences' rows of the tile add exactly 0.
//
// GQA: query heads come in groups sharing a K/V head (args.group > 1); an item
// then walks the query tiles of its whole group.
template <int D, typename VT, bool GQA, int KBUFS>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dqa, const __grid_constant__ BwdArgs args,
               const __grid_constant__ VT vt) {
  constexpr bool VARLEN = std::is_same_v<VT, VarlenTable>;
  constexpr bool PACKED = std::is_same_v<VT, PackedTiles>;
  using L = BwdSmem<D, KBUFS>;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  if (!L::kAlignSlack && (raw & 1023u) != 0) {
    // No slack to realign (see BwdSmem): report and leave before touching anything.
    pdl_wait();
    if (threadIdx.x == 0) atomicExch(args.status, DEV_SMEM_ALIGN);
    return;
  }
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H_kv = args.H_kv;
  int n_items;
  if constexpr (VARLEN)
    n_items = vt.total * H_kv;
  else if constexpr (PACKED)
    n_items = (vt.n_seqs + vt.pack - 1) / vt.pack;
  else
    n_items = args.B * H_kv * args.n_ktiles;
  // 128-row box (or 32-column fp32 box for the dQ reduce) whose first row is
  // `row` of head `head`.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* m, uint32_t bar, int col, int row, int head) {
    if constexpr (VARLEN)
      tma_load_3d(dst, m, bar, col, head, row);
    else
      tma_load_3d(dst, m, bar, col, row, head);
  };
  auto reduce_rows = [&](uint32_t src, int col, int row, int head) {
    if constexpr (VARLEN)
      tma_reduce_add_3d(&tm_dqa, src, col, head, row);
    else
      tma_reduce_add_3d(&tm_dqa, src, col, row, head);
  };

  const uint32_t sSt = sbase + L::offStage;
  const uint32_t sDS = sbase + L::offDS;
  const uint32_t sK = sbase + L::offK, sV = sbase + L::offV;
  const uint32_t bar0 = sbase + L::offBar;
  // K is read until an item's last dQ MMA, V only until its last dP^T MMA
  // (early in the last tile), so each has its own barriers and the next
  // item's V loads while the current item finishes.
  constexpr int KB = L::kKBufs;
  auto k_full = [&](int b) { return bar0 + 8u * b; };
  auto k_empty = [&](int b) { return bar0 + 8u * (KB + b); };
  const uint32_t v_full = bar0 + 8u * (2 * KB), v_empty = v_full + 8;
  auto st_full = [&](int s) { return bar0 + 8u * (2 * KB + 2 + s); };
  auto st_empty = [&](int s) { return bar0 + 8u * (2 * KB + 2 + L::kStages + s); };
  // dv_slot(s): dV of the tile in stage slot s is done (its dO is free).
  auto dv_slot = [&](int s) { return bar0 + 8u * (2 * KB + 2 + 2 * L::kStages + s); };
  const uint32_t b1 = bar0 + 8u * (2 * KB + 2 + 3 * L::kStages);
  const uint32_t s_full = b1, dp_full = b1 + 8, s_free = b1 + 16, pds_full = b1 + 24;
  const uint32_t dv_done = b1 + 32, dq_full = b1 + 40, dq_free = b1 + 48, dqs_ready = b1 + 56;
  auto mma_done = [&](int i) { return b1 + 64 + 8u * i; };  // [3]
  // ds_free: dK and dQ of the previous tile are done reading dS^T. acc_free:
  // the epilogue of the previous item has read dK and dV out of tensor memory.
  // dqs_free: the previous dQ tile's reduce has read the staging buffer.
  const uint32_t ds_free = b1 + 88, acc_free = b1 + 96, dqs_free = b1 + 104;
  // dp_free: the compute warps have loaded dP^T into registers, so the next
  // dP^T may be computed while they finish dS^T.
  const uint32_t dp_free = b1 + 112;
  const uint32_t sDQ = sbase + L::offDQ;
  // item_full(i): descriptor slot i is written; item_empty(i): every reader
  // has its copy (packed sequences only).
  auto item_full = [&](int i) { return b1 + 128 + 8u * i; };
  auto item_empty = [&](int i) { return b1 + 128 + 8u * (L::kItemRing + i); };
  // the three MMA issuer threads, the 256 compute threads and the 128 dQ threads
  constexpr int kItemReaders = 3 + 256 + 128;
  const uint32_t sItems = sbase + L::offItems;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
  const DeviceStatus st{args.status, args.limit_ns};

  if (threadIdx.x == 0) {
    for (int b = 0; b < KB; ++b) {
      mbar_init(k_full(b), 1);
      mbar_init(k_empty(b), 2);  // read by the S^T issuer and the dQ issuer
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);  // read by the dP^T issuer only
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(st_full(s), 1);
      // dV and dK are the last MMA readers of a stage; with d = 128 the
      // stage then holds the tile's dQ until the reduce has read it.
      mbar_init(st_empty(s), L::kDqInStage ? 3 : 2);
      mbar_init(dv_slot(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(s_free, 256);
    mbar_init(pds_full, 256);
    mbar_init(dv_done, 1);
    mbar_init(dq_full, 2);  // dQ (dV issuer) and dK (dK issuer) of the tile are done
    mbar_init(dq_free, 128);
    mbar_init(dqs_ready, 128);
    for (int i = 0; i < 3; ++i) mbar_init(mma_done(i), 1);
    mbar_init(ds_free, 2);  // both readers of dS^T: dK and dQ
    mbar_init(acc_free, L::kEpiOnDq ? 128 : 256);  // once dK, dV have been read out
    mbar_init(dqs_free, 1);
    mbar_init(dp_free, 256);
    if constexpr (VARLEN)
      for (int i = 0; i < L::kItemRing; ++i) {
        mbar_init(item_full(i), 1);
        mbar_init(item_empty(i), kItemReaders);
      }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpLoad) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  // Descriptor words (only the low word, start address >> 4, varies).
  constexpr uint32_t hi = sdesc_hi(1024);
  auto stage_q = [&](int g) { return sSt + (g % L::kStages) * L::kStage; };
  auto stage_do = [&](int g) { return sSt + (g % L::kStages) * L::kStage + L::kTile; };
  // K-major A and B over a 64-element-wide atom pair: K step kk.
  auto kmaj = [&](uint32_t base, int kk) {
    return sdesc_join(sdesc_lo(base, 16) + (((kk >> 2) * L::kAtom + (kk & 3) * 32) >> 4), hi);
  };
  // MN-major operand (atoms of 64 along M/N, LBO = 16 KB): K step kk = 16 rows.
  auto mnmaj = [&](uint32_t base, int kk) {
    return sdesc_join(sdesc_lo(base, L::kAtom) + kk * (2048 >> 4), hi);
  };
  constexpr uint32_t id_s = idesc_bf16(kBM, kBN, false, false);  // S^T, dP^T
  constexpr uint32_t id_kv = idesc_bf16(kBM, D, false, true);    // dV, dK
  constexpr uint32_t id_q = idesc_bf16(kBN, D, true, true);      // dQ

  // The producer's hand-over of item m (its running index in this CTA) and
  // the readers' side; false when a wait timed out.
  auto put_item = [&](int m, const BwdItem& x) {
    const int slot = m % L::kItemRing;
    if (!mbar_wait(item_empty(slot), ((m / L::kItemRing) & 1) ^ 1, abort_flag, st)) return false;
    const uint32_t p = sItems + L::kItemBytes * slot;
    st_shared_v4(p, x.kvh, x.qh0, x.ktile, x.nq1);
    st_shared_v4(p + 16, x.nq, x.kbeg, x.kend, x.qbeg);
    st_shared_v4(p + 32, static_cast<uint32_t>(x.vbase), static_cast<uint32_t>(x.vbase >> 32), 0u, 0u);
    mbar_arrive(item_full(slot));
    return true;
  };
  auto get_item = [&](int m, BwdItem& x) {
    const int slot = m % L::kItemRing;
    if (!mbar_wait(item_full(slot), (m / L::kItemRing) & 1, abort_flag, st)) return false;
    const uint32_t p = sItems + L::kItemBytes * slot;
    const uint4 a = ld_shared_v4(p), b = ld_shared_v4(p + 16), c = ld_shared_v4(p + 32);
    x.kvh = a.x;
    x.qh0 = a.y;
    x.ktile = a.z;
    x.nq1 = a.w;
    x.nq = b.x;
    x.kbeg = b.y;
    x.kend = b.z;
    x.qbeg = b.w;
    x.vbase = static_cast<size_t>(c.x) | (static_cast<size_t>(c.y) << 32);
    mbar_arrive(item_empty(slot));
    return true;
  };

  if (warp >= kWarpIssue) {
   regs_decrease<kRegsIssue>();
   if (warp == kWarpLoad && lane == 0) {
    // ---------------- TMA producer ----------------
    // Per item n (running index over items with query tiles): K into buffer
    // n % KB, V, then one stage (Q_i, dO_i, -lse2_i, D_i) per query tile.
    // Two K buffers: the loads are ordered so that the next item's first tile
    // never waits for this item's end: its first stage goes out before V
    // (which waits for this item's last dP^T), and during this item, after its
    // first three stages, the next item's K is loaded into the other buffer
    // and its V is prefetched into L2. One K buffer (K can only load once this
    // item's last dQ has read it): V and K first, then the stages, as the
    // stage-first order measured 4 % slower on the d = 128 cross-attention
    // backward; the next item's K and V are prefetched into L2.
    int n = 0, gb = 0, issued = 0, nk = 0, nv = 0;  // item, its first tile; stage, K and V loads issued
    bool ok = true;
    auto key_row = [&](const BwdItem& x) { return x.kbeg + x.ktile * kBM; };
    auto load_k = [&](int m, const BwdItem& x) {  // K of item m (running index)
      const int kb = m % KB;
      if (!mbar_wait(k_empty(kb), ((m / KB) & 1) ^ 1, abort_flag, st)) return false;
      mbar_arrive_expect_tx(k_full(kb), L::kTile);
      for (int a = 0; a < D / 64; ++a)
        load_rows(sK + kb * L::kTile + a * L::kAtom, &tm_k, k_full(kb), a * 64, key_row(x), x.kvh);
      nk = m + 1;
      return true;
    };
    auto prefetch_rows = [&](const CUtensorMap* m, const BwdItem& x) {
      for (int a = 0; a < D / 64; ++a) {
        if constexpr (VARLEN)
          tma_prefetch_l2_3d(m, a * 64, x.kvh, key_row(x));
        else
          tma_prefetch_l2_3d(m, a * 64, key_row(x), x.kvh);
      }
    };
    int w = blockIdx.x;
    // Packed sequences: each item is looked up once, the next one at this
    // item's ahead_at, and handed to the other roles as the producer starts it.
    BwdItem ahead{};
    if (VARLEN && w < n_items) ahead = bwd_item(args, vt, w);
    if (KB == 2 && w < n_items) ok = load_k(0, VARLEN ? ahead : bwd_item(args, vt, w));
    while (w < n_items && ok) {
      const BwdItem it = VARLEN ? ahead : bwd_item(args, vt, w);
      if (VARLEN && !(ok = put_item(n, it))) break;
      const int wn = w + gridDim.x;
      // The next item's K (and V) go out after this item's first three stages.
      const int ahead_at = min(2, it.nq - 1);
      QCursor<GQA> qc;
      if (KB == 1) {
        if (!(ok = mbar_wait(v_empty, (n & 1) ^ 1, abort_flag, st))) break;
        mbar_arrive_expect_tx(v_full, L::kTile);
        for (int a = 0; a < D / 64; ++a)
          load_rows(sV + a * L::kAtom, &tm_v, v_full, a * 64, key_row(it), it.kvh);
        nv = n + 1;
        if (!(ok = load_k(n, it))) break;
      }
      for (int i = 0; i < it.nq; ++i, qc.next(it)) {
        const int g = gb + i;
        const int s = g % L::kStages;
        if (!(ok = mbar_wait(st_empty(s), ((g / L::kStages) & 1) ^ 1, abort_flag, st))) break;
        const uint32_t base = sSt + s * L::kStage;
        const int qrow = qc.row(it), qhead = qc.head(it);
        const size_t voff = qc.voff(it, args.Lq_pad);
        mbar_arrive_expect_tx(st_full(s), L::kStage);
        for (int a = 0; a < D / 64; ++a) {
          load_rows(base + a * L::kAtom, &tm_q, st_full(s), a * 64, qrow, qhead);
          load_rows(base + L::kTile + a * L::kAtom, &tm_do, st_full(s), a * 64, qrow, qhead);
        }
        bulk_load(base + 2 * L::kTile, args.nlse2 + voff, L::kVec, st_full(s));
        bulk_load(base + 2 * L::kTile + L::kVec, args.delta + voff, L::kVec, st_full(s));
        issued = g + 1;
        if (i == 0 && KB == 2) {
          // V of this item once the previous item's last dP^T has read the
          // buffer; with one K buffer, K once its last dQ has.
          if (!(ok = mbar_wait(v_empty, (n & 1) ^ 1, abort_flag, st))) break;
          mbar_arrive_expect_tx(v_full, L::kTile);
          for (int a = 0; a < D / 64; ++a)
            load_rows(sV + a * L::kAtom, &tm_v, v_full, a * 64, key_row(it), it.kvh);
          nv = n + 1;
        }
        if (i == ahead_at && wn < n_items) {
          const BwdItem nx = bwd_item(args, vt, wn);
          if constexpr (VARLEN) ahead = nx;
          if (KB == 2) {
            if (!(ok = load_k(n + 1, nx))) break;
          } else {
            prefetch_rows(&tm_k, nx);
          }
          prefetch_rows(&tm_v, nx);
        }
      }
      ++n;
      gb += it.nq;
      w = wn;
    }
    // Every copy started here must land before the CTA may exit.
    for (int m = max(0, nk - KB); m < nk; ++m) mbar_wait_drain(k_full(m % KB), (m / KB) & 1, st);
    if (nv > 0) mbar_wait_drain(v_full, (nv - 1) & 1, st);
    for (int g = max(0, issued - L::kStages); g < issued; ++g)
      mbar_wait_drain(st_full(g % L::kStages), (g / L::kStages) & 1, st);
   } else if ((warp == kWarpSdp || warp == kWarpDvDq || warp == kWarpDk) && lane == 0) {
    // ---------------- MMA issuers ----------------
    // role 0 S/dP, 1 dV and dQ, 2 dK
    const int role = warp - kWarpSdp - (warp == kWarpDk ? 1 : 0);
    bool ok = true;
    int n = 0, gb = 0;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int nq;
      if constexpr (VARLEN) {
        BwdItem x;
        if (!(ok = get_item(n, x))) break;
        nq = x.nq;
      } else {
        nq = bwd_item(args, vt, w).nq;
      }
      const uint32_t sKn = sK + (n % KB) * L::kTile;  // this item's K
      // K: the S^T product (role 0) reads it from the first tile on; the dQ
      // product (role 1) waits for it before its first dQ, not before dV.
      if (role == 0 && !(ok = mbar_wait(k_full(n % KB), (n / KB) & 1, abort_flag, st))) break;
      if (role == 1 && n > 0) {
        // dV of the first tile overwrites the accumulator: the previous item's
        // epilogue must have read it.
        if (!(ok = mbar_wait(acc_free, (n - 1) & 1, abort_flag, st))) break;
      }
      for (int i = 0; i < nq && ok; ++i) {
        const int g = gb + i;
        const uint32_t ph = g & 1;
        const int s = g % L::kStages;
        const uint32_t sph = (g / L::kStages) & 1;
        if (!(ok = mbar_wait(st_full(s), sph, abort_flag, st))) break;
        if (role == 0) {
          // S^T_g = K Q_g^T into S^T, once the compute warps have read S^T_{g-1}
          // (and, when P^T lives in those columns, dV_{g-1} has read P^T_{g-1}).
          if (g > 0 && !(ok = mbar_wait(s_free, (g - 1) & 1, abort_flag, st))) break;
          if (L::kPAlias && g > 0 && !(ok = mbar_wait(dv_done, (g - 1) & 1, abort_flag, st))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + L::cS, kmaj(sKn, kk), kmaj(stage_q(g), kk), id_s, kk > 0);
          mma_commit(s_full);
          if (i == nq - 1) mma_commit(k_empty(n % KB));  // this thread's last read of K
          // dP^T_g = V dO_g^T, once dP^T_{g-1} has been read (and, when dQ
          // shares those columns, dQ_{g-1} too).
          if (g > 0) {
            if (!(ok = mbar_wait(dp_free, (g - 1) & 1, abort_flag, st))) break;
            if (L::kDqAlias && !(ok = mbar_wait(dq_free, (g - 1) & 1, abort_flag, st))) break;
          }
          if (i == 0 && !(ok = mbar_wait(v_full, n & 1, abort_flag, st))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + L::cDP, kmaj(sV, kk), kmaj(stage_do(g), kk), id_s, kk > 0);
          mma_commit(dp_full);
          if (i == nq - 1) mma_commit(v_empty);
        } else if (role == 1) {
          // dV += P^T_g dO_g once P^T_g is written.
          if (!(ok = mbar_wait(s_free, ph, abort_flag, st))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + L::cDV, tmem + L::p_col(kk), mnmaj(stage_do(g), kk), id_kv, acc);
          }
          mma_commit(dv_done);
          mma_commit(st_empty(s));
          if constexpr (L::kDqInStage) mma_commit(dv_slot(s));
          // dQ_g = dS_g K once dS^T_g is written and dQ_{g-1} has been read out
          // of tensor memory (issued here, beside dV, so that dK and dQ go out
          // from two threads and dS^T is released sooner).
          if (!(ok = mbar_wait(pds_full, ph, abort_flag, st))) break;
          if (g > 0 && !(ok = mbar_wait(dq_free, (g - 1) & 1, abort_flag, st))) break;
          if (i == 0 && !(ok = mbar_wait(k_full(n % KB), (n / KB) & 1, abort_flag, st))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ss(tmem + L::cDQ, mnmaj(sDS, kk), mnmaj(sKn, kk), id_q, kk > 0);
          mma_commit(dq_full);
          mma_commit(ds_free);
          if (i == nq - 1) mma_commit(k_empty(n % KB));  // this thread's last read of K
        } else {
          // dK += dS^T_g Q_g once dS^T_g is written (for the first tile's dK,
          // once the previous item's dK has been read out).
          if (!(ok = mbar_wait(pds_full, ph, abort_flag, st))) break;
          if (i == 0 && n > 0 && !(ok = mbar_wait(acc_free, (n - 1) & 1, abort_flag, st))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ss(tmem + L::cDK, kmaj(sDS, kk), mnmaj(stage_q(g), kk), id_kv,
                   (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(dq_full);
          mma_commit(st_empty(s));
          mma_commit(ds_free);
        }
      }
      ++n;
      gb += nq;
    }
    // Every MMA this thread issued must be finished before tensor memory is released.
    mma_commit(mma_done(role));
    mbar_wait_drain(mma_done(role), 0, st);
   }
  } else if (warp >= kWarpDq) {
    regs_decrease<kRegsDq>();
    // ---------------- dQ warpgroup ----------------
    const int sub = warp & 3;
    const int r = sub * 32 + lane;
    const bool leader = (r == 0);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const uint32_t tq = lane_base + L::cDQ;
    bool ok = true;
    int gb = 0, m = 0;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++m) {
      BwdItem it;
      if constexpr (VARLEN) {
        if (!(ok = __all_sync(0xffffffffu, get_item(m, it)))) break;
      } else {
        it = bwd_item(args, vt, w);
      }
      QCursor<GQA> qc;
      for (int i = 0; i < it.nq && ok; ++i, qc.next(it)) {
        const int g = gb + i;
        const int qrow = qc.row(it), qhead = qc.head(it);
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(dq_full, g & 1, abort_flag, st)))) break;
        tc_fence_after();
        if (L::kEpiOnDq && i == it.nq - 1) {
          // ---------------- dK, dV epilogue of the item ----------------
          // dq_full of the item's last tile means its dK is done; with dV
          // done too, key row r of both accumulators goes out as bf16 rows of
          // dV and dK (dK scaled), 32 columns at a time, and acc_free lets
          // the next item's first dV and dK overwrite them. Done here, not by
          // the compute warps, so those start the next item's first tile
          // straight away.
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(dv_done, g & 1, abort_flag, st)))) break;
          tc_fence_after();
          const int key = it.kbeg + it.ktile * kBM + r;
          const bool key_ok = key < it.kend;
          // element offset of this key row of dK, dV: [B*H_kv, Lk, d], or token-major [T, H_kv, d]
          const size_t k_off = VARLEN ? (static_cast<size_t>(key) * H_kv + it.kvh) * D
                                      : (static_cast<size_t>(it.kvh) * args.Lk + key) * D;
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const float mul = which == 0 ? 1.f : args.scale;
            uint4* dst = reinterpret_cast<uint4*>(
                static_cast<__nv_bfloat16*>(which == 0 ? args.dv : args.dk) + k_off);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t x[32];
              tmem_ld32(lane_base + (which == 0 ? L::cDV : L::cDK) + 32 * c, x);
              tmem_wait_ld();
              reg_pin(x);
              if (which == 1 && c == D / 32 - 1) {
                tc_fence_before();
                mbar_arrive(acc_free);  // the next item's first dV / dK may overwrite them
              }
              if (key_ok) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const uint32_t* y = x + 8 * u;
                  dst[4 * c + u] = make_uint4(
                      pack_bf16(__uint_as_float(y[0]) * mul, __uint_as_float(y[1]) * mul),
                      pack_bf16(__uint_as_float(y[2]) * mul, __uint_as_float(y[3]) * mul),
                      pack_bf16(__uint_as_float(y[4]) * mul, __uint_as_float(y[5]) * mul),
                      pack_bf16(__uint_as_float(y[6]) * mul, __uint_as_float(y[7]) * mul));
                }
              }
            }
          }
        }
        if constexpr (PACKED) {
          // Packed short sequences: every query row of the tile gets its whole
          // dQ here (its sequence's keys are all in this key tile), so it is
          // scaled and stored as bf16 directly, with no fp32 accumulator.
          const int ns = min(vt.pack, vt.n_seqs - w * vt.pack);
          const bool row_ok = r < ns * vt.Lq;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.dq) +
                                                static_cast<size_t>(qrow + r) * D);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tq + 32 * c, v);
            tmem_wait_ld();
            reg_pin(v);
            if (c == D / 32 - 1) {
              tc_fence_before();
              mbar_arrive(dq_free);  // the TMEM dQ tile may be overwritten now
            }
            if (row_ok) {
              const float sc = args.scale;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t* x = v + 8 * u;
                dst[4 * c + u] = make_uint4(
                    pack_bf16(__uint_as_float(x[0]) * sc, __uint_as_float(x[1]) * sc),
                    pack_bf16(__uint_as_float(x[2]) * sc, __uint_as_float(x[3]) * sc),
                    pack_bf16(__uint_as_float(x[4]) * sc, __uint_as_float(x[5]) * sc),
                    pack_bf16(__uint_as_float(x[6]) * sc, __uint_as_float(x[7]) * sc));
              }
            }
          }
          // The stage slot is not used for dQ here; release its dQ share.
          if (L::kDqInStage && leader) mbar_arrive(st_empty(g % L::kStages));
        } else if constexpr (!L::kDqInStage) {
          uint32_t v0[32], v1[32];
          tmem_ld32(tq, v0);
          tmem_ld32(tq + 32, v1);
          tmem_wait_ld();
          reg_pin(v0);
          reg_pin(v1);
          tc_fence_before();
          mbar_arrive(dq_free);  // the TMEM dQ tile may be overwritten now
          // The previous tile's reduce must have finished reading the staging buffer.
          if (g > 0 &&
              !(ok = __all_sync(0xffffffffu, mbar_wait(dqs_free, (g - 1) & 1, abort_flag, st))))
            break;
          // Row r -> two 128-byte-swizzled [128 x 32] fp32 boxes.
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            st_shared_v4(sDQ + sw128_offset(r, ch), v0[4 * ch], v0[4 * ch + 1], v0[4 * ch + 2],
                         v0[4 * ch + 3]);
            st_shared_v4(sDQ + L::kAtom + sw128_offset(r, ch), v1[4 * ch], v1[4 * ch + 1],
                         v1[4 * ch + 2], v1[4 * ch + 3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(dqs_ready);
          if (leader) {
            if (!mbar_wait(dqs_ready, g & 1, abort_flag, st)) {
              ok = false;
            } else {
              reduce_rows(sDQ, 0, qrow, qhead);
              reduce_rows(sDQ + L::kAtom, 32, qrow, qhead);
              bulk_commit_group();
              bulk_wait_group_read0();
              mbar_arrive(dqs_free);
            }
          }
          ok = __all_sync(0xffffffffu, ok);
        } else {
          // The tile's stage slot takes its dQ: dK_g and dQ_g (Q_g) are done
          // (dq_full), dV_g (dO_g) once dv_slot says so. Row r -> four
          // 128-byte-swizzled [128 x 32] fp32 boxes over the 64 KB slot.
          const int s = g % L::kStages;
          if (!(ok = __all_sync(0xffffffffu,
                                mbar_wait(dv_slot(s), (g / L::kStages) & 1, abort_flag, st))))
            break;
          const uint32_t sDQs = sSt + s * L::kStage;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tq + 32 * c, v);
            tmem_wait_ld();
            reg_pin(v);
            if (c == D / 32 - 1) {
              tc_fence_before();
              mbar_arrive(dq_free);  // the TMEM dQ tile may be overwritten now
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              st_shared_v4(sDQs + c * L::kAtom + sw128_offset(r, ch), v[4 * ch], v[4 * ch + 1],
                           v[4 * ch + 2], v[4 * ch + 3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(dqs_ready);
          if (leader) {
            if (!mbar_wait(dqs_ready, g & 1, abort_flag, st)) {
              ok = false;
            } else {
#pragma unroll
              for (int c = 0; c < D / 32; ++c)
                reduce_rows(sDQs + c * L::kAtom, 32 * c, qrow, qhead);
              bulk_commit_group();
              bulk_wait_group_read0();
              mbar_arrive(st_empty(s));  // the producer may reload the slot
            }
          }
          ok = __all_sync(0xffffffffu, ok);
        }
      }
      gb += it.nq;
    }
    // Reduce-adds in flight must complete before the CTA exits.
    if (leader) bulk_wait_group0();
  } else {
    regs_increase<kRegsCompute>();
    // ---------------- compute warpgroups ----------------
    const int wg = warp >> 2;  // query-column half
    const int sub = warp & 3;
    const int r = sub * 32 + lane;  // key row within the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const float sl2 = args.scale_log2;
    bool ok = true;
    int gb = 0;
    int m = 0;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++m) {
      BwdItem it;
      if constexpr (VARLEN) {
        if (!(ok = __all_sync(0xffffffffu, get_item(m, it)))) break;
      } else {
        it = bwd_item(args, vt, w);
      }
      const int nq = it.nq;
      const int key = it.kbeg + it.ktile * kBM + r;
      const bool key_ok = key < it.kend;
      // element offset of this key row of dK, dV: [B*H_kv, Lk, d], or token-major [T, H_kv, d]
      const size_t k_off = VARLEN ? (static_cast<size_t>(key) * H_kv + it.kvh) * D
                                  : (static_cast<size_t>(it.kvh) * args.Lk + key) * D;
      for (int i = 0; i < nq && ok; ++i) {
        const int g = gb + i;
        const uint32_t ph = g & 1;
        const uint32_t stg = sSt + (g % L::kStages) * L::kStage;
        const float4* nlse2_s =
            reinterpret_cast<const float4*>(smem + (stg - sbase) + 2 * L::kTile) + 16 * wg;
        const float4* dlt_s = nlse2_s + kBN / 4;
        // -lse2_g and D_g arrive with the stage's TMA copies.
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(st_full(g % L::kStages),
                                                     (g / L::kStages) & 1, abort_flag, st))))
          break;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full, ph, abort_flag, st)))) break;
        tc_fence_after();
        // P^T for this warpgroup's 64 query columns, rounded to bf16 and kept
        // packed: the same values feed dV = P^T dO and dS = P * (dP - D).
        // P^T for this warpgroup's 64 query columns: pf in fp32 (for dS), pp
        // rounded to bf16 and packed (the A operand of dV).
        uint32_t pp[32];
        float pf[64];
        {
          // Staged so that each step has 32-64 independent operations: -lse2 of
          // the 64 columns, S^T from TMEM, x = s * scale * log2e - lse2, 2^x, pack.
          float4 l4[16];
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) l4[j4] = nlse2_s[j4];
          uint32_t rr[64];
          tmem_ld32(lane_base + L::cS + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(rr));
          tmem_ld32(lane_base + L::cS + 64 * wg + 32, *reinterpret_cast<uint32_t(*)[32]>(rr + 32));
          tmem_wait_ld();
          reg_pin(*reinterpret_cast<uint32_t(*)[32]>(rr));
          reg_pin(*reinterpret_cast<uint32_t(*)[32]>(rr + 32));
          const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const float2 a = fma2(make_float2(__uint_as_float(rr[4 * j4]), __uint_as_float(rr[4 * j4 + 1])),
                                  sl2v, make_float2(l4[j4].x, l4[j4].y));
            const float2 b = fma2(make_float2(__uint_as_float(rr[4 * j4 + 2]), __uint_as_float(rr[4 * j4 + 3])),
                                  sl2v, make_float2(l4[j4].z, l4[j4].w));
            pf[4 * j4] = a.x;
            pf[4 * j4 + 1] = a.y;
            pf[4 * j4 + 2] = b.x;
            pf[4 * j4 + 3] = b.y;
          }
          if constexpr (PACKED) {
            // Block-diagonal: this key row's own sequence's queries, in this
            // warpgroup's columns [lo, hi).
            const int lo = (r / vt.Lk) * vt.Lq - 64 * wg, hi = lo + vt.Lq;
#pragma unroll
            for (int j = 0; j < 64; ++j) pf[j] = (key_ok && j >= lo && j < hi) ? ex2_approx(pf[j]) : 0.f;
          } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) pf[j] = key_ok ? ex2_approx(pf[j]) : 0.f;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) pp[j] = pack_bf16(pf[2 * j], pf[2 * j + 1]);
        }
        // dV_{g-1} must be done reading P^T before it is overwritten.
        if (g > 0) {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(dv_done, (g - 1) & 1, abort_flag, st))))
            break;
          tc_fence_after();
        }
        tmem_st32(lane_base + L::p_store_col(wg), pp);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(s_free);

        if (!(ok = __all_sync(0xffffffffu, mbar_wait(dp_full, ph, abort_flag, st)))) break;
        tc_fence_after();
        // dS = P * (dP - D) for the 64 columns, 32 at a time, on packed fp32
        // pairs with the fp32 P (dV uses P rounded to bf16; the rounding only
        // exists because P is a bf16 MMA operand there).
        uint32_t dsp[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float4 d4[8];
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) d4[j4] = dlt_s[8 * h + j4];
          uint32_t rr[32];
          tmem_ld32(lane_base + L::cDP + 64 * wg + 32 * h, rr);
          tmem_wait_ld();
          reg_pin(rr);
          if (h == 1) {
            tc_fence_before();
            mbar_arrive(dp_free);  // dP^T_g is in registers: dP^T_{g+1} may overwrite it
          }
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float* pj = pf + 32 * h + 4 * j4;
            const float2 a = mul2(make_float2(pj[0], pj[1]),
                                  sub2(make_float2(__uint_as_float(rr[4 * j4]), __uint_as_float(rr[4 * j4 + 1])),
                                       make_float2(d4[j4].x, d4[j4].y)));
            const float2 b = mul2(make_float2(pj[2], pj[3]),
                                  sub2(make_float2(__uint_as_float(rr[4 * j4 + 2]), __uint_as_float(rr[4 * j4 + 3])),
                                       make_float2(d4[j4].z, d4[j4].w)));
            dsp[16 * h + 2 * j4] = pack_bf16(a.x, a.y);
            dsp[16 * h + 2 * j4 + 1] = pack_bf16(b.x, b.y);
          }
        }
        // dK_{g-1} and dQ_{g-1} must be done reading dS^T before it is overwritten.
        if (g > 0 &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (g - 1) & 1, abort_flag, st))))
          break;
        const uint32_t drow = sDS + wg * L::kAtom;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(drow + sw128_offset(r, ch), dsp[4 * ch], dsp[4 * ch + 1], dsp[4 * ch + 2],
                       dsp[4 * ch + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(pds_full);
      }
      if constexpr (!L::kEpiOnDq) {
        if (!ok) break;
        // ---------------- dK, dV epilogue of the item ----------------
        // The last dV and dK (dq_full comes after both dK and dQ of a tile)
        // of the item; every earlier phase of these barriers has completed.
        const int gl = gb + nq - 1;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(dv_done, gl & 1, abort_flag, st) &&
                                               mbar_wait(dq_full, gl & 1, abort_flag, st))))
          break;
        tc_fence_after();
        uint32_t vv[D / 2], kv[D / 2];
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tmem_ld32(lane_base + L::cDV + (D / 2) * wg + 32 * c,
                    *reinterpret_cast<uint32_t(*)[32]>(vv + 32 * c));
          tmem_ld32(lane_base + L::cDK + (D / 2) * wg + 32 * c,
                    *reinterpret_cast<uint32_t(*)[32]>(kv + 32 * c));
        }
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          reg_pin(*reinterpret_cast<uint32_t(*)[32]>(vv + 32 * c));
          reg_pin(*reinterpret_cast<uint32_t(*)[32]>(kv + 32 * c));
        }
        tc_fence_before();
        mbar_arrive(acc_free);  // the next item's first dV / dK may overwrite them
        if (key_ok) {
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const uint32_t* src = which == 0 ? vv : kv;
            const float mul = which == 0 ? 1.f : args.scale;
            uint4* dst = reinterpret_cast<uint4*>(
                static_cast<__nv_bfloat16*>(which == 0 ? args.dv : args.dk) + k_off + (D / 2) * wg);
#pragma unroll
            for (int u = 0; u < D / 16; ++u) {
              const uint32_t* x = src + 8 * u;
              dst[u] = make_uint4(
                  pack_bf16(__uint_as_float(x[0]) * mul, __uint_as_float(x[1]) * mul),
                  pack_bf16(__uint_as_float(x[2]) * mul, __uint_as_float(x[3]) * mul),
                  pack_bf16(__uint_as_float(x[4]) * mul, __uint_as_float(x[5]) * mul),
                  pack_bf16(__uint_as_float(x[6]) * mul, __uint_as_float(x[7]) * mul));
            }
          }
        }
      }
      gb += nq;
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpLoad) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// D_i = sum_k dO_ik O_ik and -lse2_i = -lse_i * log2(e) (stored negated, the
// addend of the exponent) for rows < Lq; padding rows up to the 128-row tile
// boundary get D = 0 and -lse2 = -inf (so their
// recomputed P is exactly 0). Also zeroes the fp32 dQ accumulator.
// VarlenTable: each sequence's rows are padded to whole tiles (padded row p
// of a head is row p - 128 cu_qt[s] of the sequence s owning tile p / 128).
// PackedTiles: padded row p is row p % 128 of tile p / 128, which holds the
// query rows of that tile's sequences (flattened row i * pack * Lq + p % 128).
template <int D, typename VT>
__global__ void __launch_bounds__(256)
    bwd_pre_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ VT vt) {
  constexpr bool VARLEN = std::is_same_v<VT, VarlenTable>;
  constexpr bool PACKED = std::is_same_v<VT, PackedTiles>;
  constexpr int kLanesPerRow = D / 8;  // 16 bytes of bf16 per lane
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  pdl_launch_dependents();
  pdl_wait();
  const long long gwarp = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  const long long prow = gwarp * kRowsPerWarp + lane / kLanesPerRow;  // padded row index
  const int seg = lane % kLanesPerRow;
  const long long total = static_cast<long long>(a.B) * a.H * a.Lq_pad;
  const bool in_range = prow < total;
  const long long bh = in_range ? prow / a.Lq_pad : 0;
  int r = in_range ? static_cast<int>(prow - bh * a.Lq_pad) : a.Lq;  // query row (token)
  bool valid;
  size_t off;  // element offset of the row's 8-column segment in O, dO and the dQ accumulator
  if constexpr (VARLEN) {
    valid = false;
    if (in_range) {
      const int s = seq_of(vt.cu_qt, vt.n_seqs, r / kBN);
      const int rr = r - vt.cu_qt[s] * kBN;
      valid = rr < vt.cu_q[s + 1] - vt.cu_q[s];
      r = vt.cu_q[s] + rr;
    }
    off = (static_cast<size_t>(r) * a.H + bh) * D + seg * 8;
  } else if constexpr (PACKED) {
    // B = H = 1 here: bh = 0 and r is the padded row
    valid = false;
    if (in_range) {
      const int i = r / kBN, rr = r - i * kBN;
      valid = rr < min(vt.pack, vt.n_seqs - i * vt.pack) * vt.Lq;
      r = i * vt.pack * vt.Lq + rr;
    }
    off = static_cast<size_t>(r) * D + seg * 8;
  } else {
    valid = in_range && r < a.Lq;
    off = (static_cast<size_t>(bh) * a.Lq + r) * D + seg * 8;
  }
  float dot = 0.f;
  if (valid) {
    const uint4 o4 = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.o) + off);
    const uint4 d4 = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dO) + off);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o4);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d4);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 of = __bfloat1622float2(o2[u]);
      const float2 df = __bfloat1622float2(d2[u]);
      dot = fmaf(of.x, df.x, dot);
      dot = fmaf(of.y, df.y, dot);
    }
    if constexpr (!PACKED) {  // packed tiles store dQ directly: no accumulator
      float4* z = reinterpret_cast<float4*>(a.dq_acc + off);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int m = kLanesPerRow / 2; m > 0; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
  if (in_range && seg == 0) {
    a.delta[prow] = valid ? dot : 0.f;
    a.nlse2[prow] = valid ? -(a.lse[bh * a.Lq + r] * kLog2e) : -INFINITY;
  }
}

__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ acc,
                                                     __nv_bfloat16* __restrict__ dq, float scale,
                                                     long long n8) {
  pdl_launch_dependents();
  pdl_wait();
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= n8) return;
  const float4 a0 = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * i);
  const float4 a1 = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
  reinterpret_cast<uint4*>(dq)[i] =
      make_uint4(pack_bf16(a0.x * scale, a0.y * scale), pack_bf16(a0.z * scale, a0.w * scale),
                 pack_bf16(a1.x * scale, a1.y * scale), pack_bf16(a1.z * scale, a1.w * scale));
}

template <int D, typename VT, bool GQA, int KBUFS>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a,
                         const VT& vt, long long items, cudaStream_t stream) {
  using L = BwdSmem<D, KBUFS>;
  {
    constexpr int kRowsPerBlock = 8 * (32 / (D / 8));
    const long long total = static_cast<long long>(a.B) * a.H * a.Lq_pad;
    const long long blocks = (total + kRowsPerBlock - 1) / kRowsPerBlock;
    cudaError_t e = launch_pdl(bwd_pre_kernel<D, VT>, dim3(static_cast<unsigned>(blocks)),
                               dim3(256), 0, stream, a, vt);
    if (e != cudaSuccess) return e;
  }
  if (items > 0) {
    auto kern = bwd_kernel<D, VT, GQA, KBUFS>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    // The warpgroups' register shares must fit the launch allocation, or an
    // increase would wait forever: refuse to launch otherwise.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kRegsAtLaunch) return cudaErrorInvalidConfiguration;
    // Persistent: one CTA per SM (tensor memory and shared memory allow no
    // more), each walking its share of the work items.
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), L::kAlloc, stream, tq, tk, tv, tdo, tdqa, a,
                   vt);
    if (e != cudaSuccess) return e;
  }
  if (!std::is_same_v<VT, PackedTiles>) {  // packed tiles wrote bf16 dQ already
    const long long n8 = static_cast<long long>(a.B) * a.H * a.Lq * D / 8;
    const long long blocks = (n8 + 255) / 256;
    return launch_pdl(bwd_dq_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                      a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), a.scale, n8);
  }
  return cudaSuccess;
}

// Items of at most 32 query tiles (on average) take the two-K-buffer form at
// d = 64 (see BwdSmem), except packed sequences: with their items handed
// over by the producer, one K buffer measured faster on both the packed mix
// of 196- to 1568-token sequences (backward 454 -> 443 us) and 16 sequences
// of 1568 tokens (532 -> 515 us).
template <int D, typename VT, bool GQA = false>
cudaError_t launch_bwd_k(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a,
                         const VT& vt, long long items, double tiles_per_item,
                         cudaStream_t stream) {
  if constexpr (D == 64 && !std::is_same_v<VT, VarlenTable>)
    if (tiles_per_item <= 32.0)
      return launch_bwd_t<D, VT, GQA, 2>(tq, tk, tv, tdo, tdqa, a, vt, items, stream);
  return launch_bwd_t<D, VT, GQA, 1>(tq, tk, tv, tdo, tdqa, a, vt, items, stream);
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a, int d,
                       cudaStream_t stream) {
  const long long items = static_cast<long long>(a.n_ktiles) * a.B * a.H_kv;
  const double tpi = static_cast<double>(a.group) * a.n_qtiles;
  const NoVarlen nv{};
  if (a.group > 1)
    return d == 64 ? launch_bwd_k<64, NoVarlen, true>(tq, tk, tv, tdo, tdqa, a, nv, items, tpi, stream)
                   : launch_bwd_k<128, NoVarlen, true>(tq, tk, tv, tdo, tdqa, a, nv, items, tpi, stream);
  return d == 64 ? launch_bwd_k<64, NoVarlen>(tq, tk, tv, tdo, tdqa, a, nv, items, tpi, stream)
                 : launch_bwd_k<128, NoVarlen>(tq, tk, tv, tdo, tdqa, a, nv, items, tpi, stream);
}

cudaError_t launch_bwd_varlen(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a,
                              const VarlenTable& vt, int d, cudaStream_t stream) {
  const long long items = static_cast<long long>(vt.total) * a.H_kv;
  // query tiles per item, averaged over the items (a sequence's key tiles
  // each walk its query tiles, for every head of the group)
  double tiles = 0.0;
  for (int s = 0; s < vt.n_seqs; ++s)
    tiles += static_cast<double>(vt.cu_items[s + 1] - vt.cu_items[s]) * (vt.cu_qt[s + 1] - vt.cu_qt[s]);
  const double tpi = vt.total > 0 ? a.group * tiles / vt.total : 0.0;
  if (a.group > 1)
    return d == 64 ? launch_bwd_k<64, VarlenTable, true>(tq, tk, tv, tdo, tdqa, a, vt, items, tpi, stream)
                   : launch_bwd_k<128, VarlenTable, true>(tq, tk, tv, tdo, tdqa, a, vt, items, tpi, stream);
  return d == 64 ? launch_bwd_k<64, VarlenTable>(tq, tk, tv, tdo, tdqa, a, vt, items, tpi, stream)
                 : launch_bwd_k<128, VarlenTable>(tq, tk, tv, tdo, tdqa, a, vt, items, tpi, stream);
}

cudaError_t launch_bwd_packed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a,
                              const PackedTiles& pt, int d, cudaStream_t stream) {
  const long long items = (static_cast<long long>(pt.n_seqs) + pt.pack - 1) / pt.pack;
  return d == 64 ? launch_bwd_k<64, PackedTiles>(tq, tk, tv, tdo, tdqa, a, pt, items, 1.0, stream)
                 : launch_bwd_k<128, PackedTiles>(tq, tk, tv, tdo, tdqa, a, pt, items, 1.0, stream);
}

}  // namespace eba
