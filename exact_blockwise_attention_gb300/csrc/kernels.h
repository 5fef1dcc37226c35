// Internal interface between the C-ABI layer (attn_api.cu) and the kernel
// translation units. Host-side only: argument blocks and launcher functions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "attn.h"

namespace eba {

// Launch with programmatic stream serialization (see pdl_wait): the kernel may
// be scheduled while the previous kernel in the stream finishes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kTileRows = 128;  // query rows per Q tile and keys per KV tile

// Device address of one of the library's __device__ variables (`symbol` is its
// host-side shadow, never a device address) in the context current on the
// calling thread (bound first if the thread has none). Looked up with
// cudaGetSymbolAddress and cached per device and context: a context
// re-created after a device reset gets a fresh lookup. nullptr on failure,
// with the CUDA error recorded for attn_last_cuda_error.
enum : int { kSymStatusWord = 0, kSymNoallocScratch = 1, kSymSlots = 2 };
void* symbol_address(const void* symbol, int slot);
// Record a CUDA error code for attn_last_cuda_error (calling thread).
void record_cuda_error(int e);

// Forward / partial-forward launch arguments (one launch may cover several
// KV chunks: grid.y = chunk).
struct FwdArgs {
  int B, H, Lq, Lk;
  int group;  // query heads per K/V head (1: multi-head; H / H_kv: grouped-query)
  int n_qtiles;  // ceil(Lq / 128)
  int n_pairs;   // ceil(n_qtiles / 2): one CTA handles two Q tiles
  int n_chunks;
  float scale_log2;  // softmax scale * log2(e) (FP8: times the Q and K dequantisation scales)
  float o_scale;     // FP8: the V dequantisation scale (O multiplier); otherwise unused
  int bounds[ATTN_MAX_CHUNKS + 1];
  void* o;     // bf16 [B,H,Lq,d] (full forward) or fp32 [C,B,H,Lq,d] (partials)
  float* lse;  // [C,B,H,Lq]
  long long o_chunk_stride;    // elements between consecutive chunks of o
  long long lse_chunk_stride;  // elements between consecutive chunks of lse
  int* status;
  unsigned long long limit_ns;
};

// Backward launch arguments.
struct BwdArgs {
  int B, H, Lq, Lk;
  int group;  // query heads per K/V head
  int H_kv;   // K/V heads: K, V, dK, dV are [B, H_kv, Lk, d] (H = group * H_kv)
  int n_qtiles, n_ktiles;
  int Lq_pad;  // n_qtiles * 128
  float scale;
  float scale_log2;
  const void* o;    // bf16 [B,H,Lq,d]
  const void* dO;   // bf16 [B,H,Lq,d]
  const float* lse; // [B,H,Lq]
  float* dq_acc;    // fp32 [B,H,Lq,d] workspace
  float* nlse2;     // fp32 [B,H,Lq_pad] workspace: -lse * log2(e), -inf on padding rows
  float* delta;     // fp32 [B,H,Lq_pad] workspace: D_i = sum_k dO_ik O_ik, 0 on padding
  void* dq;         // bf16 [B,H,Lq,d]
  void* dk;         // bf16 [B,H/group,Lk,d]
  void* dv;         // bf16 [B,H/group,Lk,d]
  int* status;
  unsigned long long limit_ns;
};

// Packed variable-length sequences (token-major [T, H, d]): the kernels' work
// items are counted per sequence, cu_items being the prefix sum of the
// sequences' item counts (forward: pairs of 128-row query tiles; backward:
// 128-row key tiles, none for a sequence without queries). cu_qt is the prefix sum of the sequences' query-tile
// counts ceil(Lq_s / 128): the backward keeps its per-row -lse2 and D with
// each sequence padded to whole tiles, tile t of the packed order at rows
// [128 t, 128 t + 128) of a head.
//
// Work items are numbered rank-major: the sequences in order of decreasing
// cost per item (rank r is sequence order[r]; the backward's items cost in
// proportion to their sequence's query tiles, the forward's to its key
// tiles), then head, then the sequence's own items; cu_rank is the prefix sum
// of the item counts in that order. With the snake dealing of varlen_pos,
// the persistent CTAs then get nearly equal work although the sequences'
// items differ in size.
struct VarlenTable {
  int n_seqs;
  int total;  // cu_items[n_seqs]
  int cu_q[ATTN_MAX_SEQS + 1];
  int cu_k[ATTN_MAX_SEQS + 1];
  int cu_items[ATTN_MAX_SEQS + 1];
  int cu_qt[ATTN_MAX_SEQS + 1];
  int order[ATTN_MAX_SEQS];
  int cu_rank[ATTN_MAX_SEQS + 1];
};
struct NoVarlen {};

#ifdef __CUDACC__
// Persistent CTAs deal the items round-robin: CTA c takes w = c + k G in round
// k (G = gridDim.x). snake_order re-deals them so that in odd rounds, unless
// the round is the last and partial, CTA c takes the round's item G - 1 - c:
// with items in order of decreasing cost the CTAs' totals even out. A
// bijection on [0, n).
__device__ __forceinline__ int snake_order(int w, int n) {
  const int G = static_cast<int>(gridDim.x);
  const int k = w / G;
  if ((k & 1) && (k + 1) * G <= n) return k * G + (G - 1) - (w - k * G);
  return w;
}

// Packed-sequence item w of `heads` heads: its sequence, head and index among
// the sequence's items (see VarlenTable).
struct VarlenPos {
  int seq, head, idx;
};
__device__ __forceinline__ VarlenPos varlen_pos(const VarlenTable& vt, int heads, int w) {
  w = snake_order(w, vt.total * heads);
  int lo = 0, hi = vt.n_seqs;  // the rank r with heads cu_rank[r] <= w < heads cu_rank[r + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (heads * vt.cu_rank[mid] <= w) lo = mid; else hi = mid;
  }
  VarlenPos p;
  p.seq = vt.order[lo];
  const int n = vt.cu_items[p.seq + 1] - vt.cu_items[p.seq];
  const int within = w - heads * vt.cu_rank[lo];
  p.head = within / n;
  p.idx = within - p.head * n;
  return p;
}
#endif

// Short sequences packed into tiles: `pack` = floor(128 / max(Lq, Lk))
// consecutive (batch, head) sequences of Lq queries and Lk keys share one
// 128-row tile of the flattened [B*H*L, d] views (tile i: sequences
// [i*pack, i*pack + pack), query rows from i*pack*Lq, key rows from
// i*pack*Lk), attended with a block-diagonal mask. Launch arguments then
// describe the flattened views: B = H = 1, Lq / Lk = total rows.
struct PackedTiles {
  int pack;    // sequences per tile (>= 2)
  int n_seqs;  // B * H
  int Lq, Lk;  // per sequence
};

struct MergeArgs {
  const float* o_parts;
  const float* lse_parts;
  int n_chunks;
  long long rows;  // B * H * Lq
  void* o;         // bf16 [rows, d]
  float* lse;      // [rows]
};

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int d, bool partial, cudaStream_t stream);
// tdqa: fp32 view of the dQ accumulator (used with d = 64: TMA reduce-add).
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a, int d,
                       cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs& a, int d, cudaStream_t stream);

// Forward over sequences of at most kShortMax queries and keys (CUDA cores).
constexpr int kShortMax = 8;
struct ShortArgs {
  const void* q;  // bf16 [n_seq, Lq, d]
  const void* k;  // bf16 [n_seq, Lk, d]
  const void* v;  // bf16 [n_seq, Lk, d]
  void* o;        // bf16 [n_seq, Lq, d]
  float* lse;     // [n_seq, Lq]
  long long n_seq;
  int Lq, Lk;     // 1 .. kShortMax
  float scale_log2;
  int* status;
  unsigned long long limit_ns;
};
cudaError_t launch_fwd_short(const ShortArgs& a, int d, cudaStream_t stream);
// Backward over the same sequences (CUDA cores; no workspace).
struct ShortBwdArgs {
  const void* q;     // bf16 [n_seq, Lq, d]
  const void* k;     // bf16 [n_seq, Lk, d]
  const void* v;     // bf16 [n_seq, Lk, d]
  const void* dO;    // bf16 [n_seq, Lq, d]
  const float* lse;  // [n_seq, Lq]
  void* dq;          // bf16 [n_seq, Lq, d]
  void* dk;          // bf16 [n_seq, Lk, d]
  void* dv;          // bf16 [n_seq, Lk, d]
  long long n_seq;
  int Lq, Lk;        // 1 .. kShortMax
  float scale, scale_log2;
  int* status;
  unsigned long long limit_ns;
};
cudaError_t launch_bwd_short(const ShortBwdArgs& a, int d, cudaStream_t stream);
// Varlen forward: FwdArgs with B = 1, Lq = Tq, Lk = Tk; maps over [T, H, d].
cudaError_t launch_fwd_varlen(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdArgs& a, const VarlenTable& vt, int d, cudaStream_t stream);
// FP8 forward (d = 128): e4m3 maps over [B*H, L, 128] (Q, K) and
// [B*H, 128, Lk] (V^T), 128 x 128 one-byte boxes.
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const FwdArgs& a, cudaStream_t stream);
// Packed short sequences; maps over the flattened [1, B*H*L, d] views.
cudaError_t launch_fwd_packed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdArgs& a, const PackedTiles& pt, int d, cudaStream_t stream);
cudaError_t launch_bwd_packed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a,
                              const PackedTiles& pt, int d, cudaStream_t stream);
// Varlen backward: BwdArgs with B = 1, Lq = Tq, Lk = Tk, Lq_pad = 128 *
// cu_qt[n_seqs] (the -lse2 / D row stride of a head); maps over [T, H, d].
cudaError_t launch_bwd_varlen(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdqa, const BwdArgs& a,
                              const VarlenTable& vt, int d, cudaStream_t stream);

}  // namespace eba
