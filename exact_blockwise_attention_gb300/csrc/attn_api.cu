// C ABI of the attention library: argument validation, TMA descriptor
// construction, the per-device status word, and kernel launches. Declarations
// and the contract of each entry point are in include/attn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "kernels.h"

namespace {

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;

std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitNs};
thread_local int t_last_cuda_error = 0;  // cudaError_t of the last failing call

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_CUDA;
}

// One status word per device, in this module's device globals (no allocation).
__device__ int g_status_word;

template <typename F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

// Make sure the calling host thread has a CUDA context bound (a fresh thread,
// e.g. an autograd worker, may have none), preferring the device whose context
// is already current. Returns the device, or -1 with the error recorded. When
// ctx_id is given it receives the bound context's process-unique ID (never
// reused, even when a context is destroyed and another is created at the same
// handle), or 0 if the driver cannot tell.
int bind_device(unsigned long long* ctx_id = nullptr) {
  using CtxGetCurrent = CUresult(CUDAAPI*)(CUcontext*);
  using CtxGetDevice = CUresult(CUDAAPI*)(CUdevice*);
  using CtxGetId = CUresult(CUDAAPI*)(CUcontext, unsigned long long*);
  static CtxGetCurrent get_ctx = driver_fn<CtxGetCurrent>("cuCtxGetCurrent");
  static CtxGetDevice get_dev = driver_fn<CtxGetDevice>("cuCtxGetDevice");
  static CtxGetId get_id = driver_fn<CtxGetId>("cuCtxGetId");
  int dev = -1;
  CUcontext ctx = nullptr;
  if (get_ctx && get_dev && get_ctx(&ctx) == CUDA_SUCCESS && ctx) {
    CUdevice d;
    if (get_dev(&d) == CUDA_SUCCESS) dev = static_cast<int>(d);
  }
  cudaError_t e = cudaSuccess;
  if (dev < 0) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);  // binds the primary context to this thread
  if (e != cudaSuccess) {
    t_last_cuda_error = static_cast<int>(e);
    return -1;
  }
  if (ctx_id) {
    *ctx_id = 0;
    ctx = nullptr;
    unsigned long long id = 0;
    if (get_ctx && get_id && get_ctx(&ctx) == CUDA_SUCCESS && ctx &&
        get_id(ctx, &id) == CUDA_SUCCESS)
      *ctx_id = id;
  }
  return dev;
}

int* status_word_ptr() {
  return static_cast<int*>(eba::symbol_address(&g_status_word, eba::kSymStatusWord));
}

}  // namespace

namespace eba {

void record_cuda_error(int e) { t_last_cuda_error = e; }

// Device addresses of the library's __device__ variables, cached per device
// and symbol together with the ID of the context they were looked up in: a
// different current context (one re-created after a device reset, say) means
// a fresh lookup, so a stale address is never handed to a kernel. Without a
// context ID from the driver every call looks the address up again.
void* symbol_address(const void* symbol, int slot) {
  struct Entry {
    unsigned long long ctx;
    void* addr;
  };
  static std::mutex mu;
  static Entry cache[kMaxDevices][kSymSlots] = {};
  unsigned long long ctx = 0;
  const int dev = bind_device(&ctx);
  if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kSymSlots) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  Entry& c = cache[dev][slot];
  if (ctx == 0 || c.ctx != ctx || !c.addr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess) {
      t_last_cuda_error = static_cast<int>(e);
      c = Entry{0, nullptr};
      return nullptr;
    }
    c = Entry{ctx, p};
  }
  return c.addr;
}

}  // namespace eba

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn =
      driver_fn<PFN_cuTensorMapEncodeTiled_v12000>("cuTensorMapEncodeTiled");
  return fn;
}

// 3-D view [B*H, L, d] of a contiguous bf16 [B, H, L, d] tensor; box of
// 64 x 128 x 1 elements (128-byte rows) with the 128-byte swizzle. Rows past L
// read as zero.
bool make_map(CUtensorMap* m, const void* ptr, long long BH, int L, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(eba::kTileRows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) t_last_cuda_error = static_cast<int>(r);
  return r == CUDA_SUCCESS;
}

// 3-D view [B*H, L, d] of a contiguous fp32 [B, H, L, d] tensor; box of
// 32 x 128 x 1 elements (128-byte rows, 128-byte swizzle), for TMA reduce-add.
bool make_map_f32(CUtensorMap* m, void* ptr, long long BH, int L, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                           static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(eba::kTileRows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) t_last_cuda_error = static_cast<int>(r);
  return r == CUDA_SUCCESS;
}

// 3-D view (d, H, T) of a contiguous token-major [T, H, d] tensor (bf16, or
// fp32 for the dQ accumulator): a box is 128 consecutive tokens of one head,
// 64 bf16 / 32 fp32 columns wide (128-byte rows, 128-byte swizzle), laid out
// in shared memory exactly like a box of the [B*H, L, d] view. Tokens past T
// read as zero.
bool make_map_thd(CUtensorMap* m, const void* ptr, long long T, int H, int d, bool f32) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t esz = f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esz,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(d) * esz};
  cuuint32_t box[3] = {f32 ? 32u : 64u, 1, static_cast<cuuint32_t>(eba::kTileRows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) t_last_cuda_error = static_cast<int>(r);
  return r == CUDA_SUCCESS;
}

// 3-D view (inner, rows, BH) of a contiguous one-byte (e4m3) tensor
// [BH, rows, inner]; box of 128 x 128 x 1 bytes with the 128-byte swizzle.
// (Q, K: inner = d = 128; V^T: inner = Lk, rows = d.) Elements past the
// extents read as zero.
bool make_map_u8(CUtensorMap* m, const void* ptr, long long BH, int rows, int inner) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(inner)};
  cuuint32_t box[3] = {128, static_cast<cuuint32_t>(eba::kTileRows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) t_last_cuda_error = static_cast<int>(r);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks packed-sequence offsets and fills the kernels' table: per sequence,
// forward items are pairs of 128-row query tiles, backward items 128-row key
// tiles. Tq, Tk: the packed totals.
int build_varlen(const int* cu_q, const int* cu_k, int n_seqs, int H, int d, float scale,
                 bool backward, eba::VarlenTable* vt, int* Tq, int* Tk) {
  if (!cu_q || !cu_k || n_seqs < 1 || H < 1) return ATTN_ERR_INVALID_ARG;
  if (n_seqs > ATTN_MAX_SEQS) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (cu_q[0] != 0 || cu_k[0] != 0) return ATTN_ERR_INVALID_ARG;
  constexpr int R = eba::kTileRows;
  vt->n_seqs = n_seqs;
  vt->cu_q[0] = vt->cu_k[0] = vt->cu_items[0] = vt->cu_qt[0] = 0;
  long long items = 0, qtiles = 0;
  for (int s = 0; s < n_seqs; ++s) {
    const int lq = cu_q[s + 1] - cu_q[s], lk = cu_k[s + 1] - cu_k[s];
    if (cu_q[s + 1] < cu_q[s] || cu_k[s + 1] < cu_k[s]) return ATTN_ERR_INVALID_ARG;
    const long long nqt = (static_cast<long long>(lq) + R - 1) / R;
    const long long nkt = (static_cast<long long>(lk) + R - 1) / R;
    qtiles += nqt;
    // a backward item is a key tile against the sequence's query tiles: a
    // sequence without queries has none (its dK, dV rows are zeroed apart)
    items += backward ? (lq > 0 ? nkt : 0) : (nqt + 1) / 2;
    if (items * H >= (1ll << 31) || qtiles * R * H >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
    vt->cu_q[s + 1] = cu_q[s + 1];
    vt->cu_k[s + 1] = cu_k[s + 1];
    vt->cu_items[s + 1] = static_cast<int>(items);
    vt->cu_qt[s + 1] = static_cast<int>(qtiles);
  }
  vt->total = static_cast<int>(items);
  // Work order: sequences by decreasing cost per item (the backward walks a
  // sequence's query tiles per item, the forward its key tiles), ties in
  // sequence order.
  int cost[ATTN_MAX_SEQS];
  for (int s = 0; s < n_seqs; ++s) {
    cost[s] = backward ? vt->cu_qt[s + 1] - vt->cu_qt[s] : (vt->cu_k[s + 1] - vt->cu_k[s] + R - 1) / R;
    vt->order[s] = s;
  }
  std::stable_sort(vt->order, vt->order + n_seqs, [&](int x, int y) { return cost[x] > cost[y]; });
  vt->cu_rank[0] = 0;
  for (int r = 0; r < n_seqs; ++r) {
    const int s = vt->order[r];
    vt->cu_rank[r + 1] = vt->cu_rank[r] + (vt->cu_items[s + 1] - vt->cu_items[s]);
  }
  *Tq = cu_q[n_seqs];
  *Tk = cu_k[n_seqs];
  if (*Tq < 1 || *Tk < 1) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

int check_sizes(int B, int H, int Lq, int Lk, int d, float scale) {
  if (B < 1 || H < 1 || Lq < 1 || Lk < 1) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p) return ATTN_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

// Short sequences (at most 64 queries and keys) are packed several to a
// 128-row tile; returns the number per tile, or 0 for the per-head tiling.
int packing(int Lq, int Lk) {
  const int L = Lq > Lk ? Lq : Lk;
  return L <= eba::kTileRows / 2 ? eba::kTileRows / L : 0;
}

int fwd_packed(const void* q, const void* k, const void* v, void* o, float* lse, long long BH,
               int Lq, int Lk, int d, int pack, float scale, void* stream) {
  int* status = status_word_ptr();
  if (!status) return ATTN_ERR_CUDA;
  if (BH * Lq >= (1ll << 31) || BH * Lk >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, 1, static_cast<int>(BH * Lq), d) ||
      !make_map(&tk, k, 1, static_cast<int>(BH * Lk), d) ||
      !make_map(&tv, v, 1, static_cast<int>(BH * Lk), d))
    return ATTN_ERR_CUDA;
  eba::FwdArgs a{};
  a.B = 1;
  a.H = 1;
  a.group = 1;
  a.Lq = static_cast<int>(BH * Lq);  // flattened rows: lse / O row = tile row + item offset
  a.Lk = static_cast<int>(BH * Lk);
  a.n_chunks = 1;
  a.bounds[0] = 0;
  a.bounds[1] = a.Lk;
  a.scale_log2 = scale * kLog2e;
  a.o = o;
  a.lse = lse;
  a.status = status;
  a.limit_ns = g_wait_limit_ns.load();
  const eba::PackedTiles pt{pack, static_cast<int>(BH), Lq, Lk};
  cudaError_t e = eba::launch_fwd_packed(tq, tk, tv, a, pt, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Sequences of at most eba::kShortMax queries and keys: the CUDA-core path.
int fwd_short(const void* q, const void* k, const void* v, void* o, float* lse, long long BH,
              int Lq, int Lk, int d, float scale, void* stream) {
  int* status = status_word_ptr();
  if (!status) return ATTN_ERR_CUDA;
  eba::ShortArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.n_seq = BH;
  a.Lq = Lq;
  a.Lk = Lk;
  a.scale_log2 = scale * kLog2e;
  a.status = status;
  a.limit_ns = g_wait_limit_ns.load();
  cudaError_t e = eba::launch_fwd_short(a, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// H_kv: K/V heads (H for multi-head attention; a divisor of H for grouped-query).
int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int H_kv, int Lq, int Lk, int d, const int* bounds, int n_chunks, float scale,
               bool partial, void* stream) {
  int* status = status_word_ptr();
  if (!status) return ATTN_ERR_CUDA;
  const long long BH = static_cast<long long>(B) * H;
  const long long BHkv = static_cast<long long>(B) * H_kv;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, BH, Lq, d) || !make_map(&tk, k, BHkv, Lk, d) ||
      !make_map(&tv, v, BHkv, Lk, d))
    return ATTN_ERR_CUDA;
  eba::FwdArgs a{};
  a.B = B;
  a.H = H;
  a.group = H / H_kv;
  a.Lq = Lq;
  a.Lk = Lk;
  a.n_qtiles = (Lq + eba::kTileRows - 1) / eba::kTileRows;
  a.n_pairs = (a.n_qtiles + 1) / 2;
  a.n_chunks = n_chunks;
  a.scale_log2 = scale * kLog2e;
  for (int c = 0; c <= n_chunks; ++c) a.bounds[c] = bounds[c];
  a.o = o;
  a.lse = lse;
  a.o_chunk_stride = BH * Lq * d;
  a.lse_chunk_stride = BH * Lq;
  a.status = status;
  a.limit_ns = g_wait_limit_ns.load();
  if (static_cast<long long>(a.n_pairs) * BH >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = eba::launch_fwd(tq, tk, tv, a, d, partial, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Lq, int Lk, int d, float scale, void* stream) {
  int s = check_sizes(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return s;
  // Sequences of 5 to 8 tokens: the CUDA-core path (8 x 8 blocks, one warp
  // each). With 4 or fewer on both sides it costs as much per sequence as an
  // 8 x 8 one, and the tensor-core tiles, packing 32 such sequences each, are
  // faster there (measured at B*H = 100352, 4 x 4, d = 64: 74 against 62 us).
  if (std::max(Lq, Lk) <= eba::kShortMax && std::max(Lq, Lk) > eba::kShortMax / 2)
    return fwd_short(q, k, v, o, lse, static_cast<long long>(B) * H, Lq, Lk, d, scale, stream);
  if (const int pack = packing(Lq, Lk))
    return fwd_packed(q, k, v, o, lse, static_cast<long long>(B) * H, Lq, Lk, d, pack, scale,
                      stream);
  const int bounds[2] = {0, Lk};
  return fwd_common(q, k, v, o, lse, B, H, H, Lq, Lk, d, bounds, 1, scale, false, stream);
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, void* o, float* lse, int B,
                 int H, int Lq, int Lk, int d, float scale, float q_scale, float k_scale,
                 float v_scale, void* stream) {
  int s = check_sizes(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  for (float f : {q_scale, k_scale, v_scale})
    if (!std::isfinite(f) || !(f > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if ((s = check_ptrs({q8, k8, vt8, o, lse})) != ATTN_OK) return s;
  if (Lk % 16 != 0) return ATTN_ERR_MISALIGNED;  // V^T rows must be 16-byte multiples
  int* status = status_word_ptr();
  if (!status) return ATTN_ERR_CUDA;
  const long long BH = static_cast<long long>(B) * H;
  CUtensorMap tq, tk, tvt;
  if (!make_map_u8(&tq, q8, BH, Lq, d) || !make_map_u8(&tk, k8, BH, Lk, d) ||
      !make_map_u8(&tvt, vt8, BH, d, Lk))
    return ATTN_ERR_CUDA;
  eba::FwdArgs a{};
  a.B = B;
  a.H = H;
  a.group = 1;
  a.Lq = Lq;
  a.Lk = Lk;
  a.n_qtiles = (Lq + eba::kTileRows - 1) / eba::kTileRows;
  a.n_pairs = (a.n_qtiles + 1) / 2;
  a.n_chunks = 1;
  a.bounds[0] = 0;
  a.bounds[1] = Lk;
  a.scale_log2 = scale * q_scale * k_scale * kLog2e;
  a.o_scale = v_scale;
  a.o = o;
  a.lse = lse;
  a.status = status;
  a.limit_ns = g_wait_limit_ns.load();
  if (static_cast<long long>(a.n_pairs) * BH >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = eba::launch_fwd_fp8(tq, tk, tvt, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int H_kv, int Lq, int Lk, int d, float scale, void* stream) {
  int s = check_sizes(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if ((s = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return s;
  if (H_kv == H) return attn_fwd(q, k, v, o, lse, B, H, Lq, Lk, d, scale, stream);
  const int bounds[2] = {0, Lk};
  return fwd_common(q, k, v, o, lse, B, H, H_kv, Lq, Lk, d, bounds, 1, scale, false, stream);
}

int attn_partial_fwd(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                     int B, int H, int Lq, int Lk, int d, int k0, int k1, float scale,
                     void* stream) {
  int s = check_sizes(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  if (k0 < 0 || k1 < k0 || k1 > Lk) return ATTN_ERR_INVALID_ARG;
  if ((s = check_ptrs({q, k, v, o_part, lse_part})) != ATTN_OK) return s;
  const int bounds[2] = {k0, k1};
  return fwd_common(q, k, v, o_part, lse_part, B, H, H, Lq, Lk, d, bounds, 1, scale, true, stream);
}

int attn_split_fwd(const void* q, const void* k, const void* v, float* o_parts, float* lse_parts,
                   int B, int H, int Lq, int Lk, int d, const int* bounds, int n_chunks,
                   float scale, void* stream) {
  int s = check_sizes(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  if (!bounds) return ATTN_ERR_INVALID_ARG;
  if (n_chunks < 1) return ATTN_ERR_INVALID_ARG;
  if (n_chunks > ATTN_MAX_CHUNKS) return ATTN_ERR_UNSUPPORTED;
  if (bounds[0] != 0 || bounds[n_chunks] != Lk) return ATTN_ERR_INVALID_ARG;
  for (int c = 0; c < n_chunks; ++c)
    if (bounds[c + 1] < bounds[c]) return ATTN_ERR_INVALID_ARG;
  if ((s = check_ptrs({q, k, v, o_parts, lse_parts})) != ATTN_OK) return s;
  return fwd_common(q, k, v, o_parts, lse_parts, B, H, H, Lq, Lk, d, bounds, n_chunks, scale, true,
                    stream);
}

size_t attn_bwd_workspace_size(int B, int H, int Lq, int Lk, int d) {
  if (check_sizes(B, H, Lq, Lk, d, 1.0f) != ATTN_OK) return 0;
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t Lq_pad = (static_cast<size_t>(Lq) + eba::kTileRows - 1) / eba::kTileRows *
                        eba::kTileRows;
  return BH * Lq * d * sizeof(float)      // dQ accumulator
         + 2 * BH * Lq_pad * sizeof(float);  // -lse2 and D
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
             float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_gqa(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, Lq, Lk, d, scale, workspace,
                      workspace_bytes, stream);
}

int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv, int Lq,
                 int Lk, int d, float scale, void* workspace, size_t workspace_bytes,
                 void* stream) {
  int s = check_sizes(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if ((s = check_ptrs({q, k, v, o, dO, lse, dq, dk, dv})) != ATTN_OK) return s;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(B, H, Lq, Lk, d))
    return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  int* status = status_word_ptr();
  if (!status) return ATTN_ERR_CUDA;
  const long long BH = static_cast<long long>(B) * H;
  const long long BHkv = static_cast<long long>(B) * H_kv;
  if (H_kv == H && std::max(Lq, Lk) <= eba::kShortMax && std::max(Lq, Lk) > eba::kShortMax / 2) {
    // Sequences of 5 to 8 tokens: the CUDA-core backward (the workspace is
    // not used; as for the forward, 4 x 4 blocks and below stay on the packed
    // tiles).
    eba::ShortBwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.dO = dO;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.n_seq = BH;
    a.Lq = Lq;
    a.Lk = Lk;
    a.scale = scale;
    a.scale_log2 = scale * kLog2e;
    a.status = status;
    a.limit_ns = g_wait_limit_ns.load();
    cudaError_t e = eba::launch_bwd_short(a, d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
  }
  CUtensorMap tq, tk, tv, tdo, tdqa;
  float* ws = static_cast<float*>(workspace);
  if (const int pack = H_kv == H ? packing(Lq, Lk) : 0) {
    // Short sequences packed into tiles over the flattened [1, B*H*L, d] views.
    if (BH * Lq >= (1ll << 31) || BH * Lk >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
    const int rq = static_cast<int>(BH * Lq), rk = static_cast<int>(BH * Lk);
    if (!make_map(&tq, q, 1, rq, d) || !make_map(&tk, k, 1, rk, d) ||
        !make_map(&tv, v, 1, rk, d) || !make_map(&tdo, dO, 1, rq, d) ||
        !make_map_f32(&tdqa, ws, 1, rq, d))
      return ATTN_ERR_CUDA;
    const eba::PackedTiles pt{pack, static_cast<int>(BH), Lq, Lk};
    const int n_tiles = static_cast<int>((BH + pack - 1) / pack);
    eba::BwdArgs a{};
    a.B = 1;
    a.H = 1;
    a.group = 1;
    a.H_kv = 1;
    a.Lq = rq;
    a.Lk = rk;
    a.Lq_pad = n_tiles * eba::kTileRows;  // -lse2 / D: 128 rows per tile
    a.scale = scale;
    a.scale_log2 = scale * kLog2e;
    a.o = o;
    a.dO = dO;
    a.lse = lse;
    a.dq_acc = ws;
    a.nlse2 = ws + static_cast<size_t>(rq) * d;
    a.delta = a.nlse2 + a.Lq_pad;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.status = status;
    a.limit_ns = g_wait_limit_ns.load();
    cudaError_t e = eba::launch_bwd_packed(tq, tk, tv, tdo, tdqa, a, pt, d,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
  }
  if (!make_map(&tq, q, BH, Lq, d) || !make_map(&tk, k, BHkv, Lk, d) ||
      !make_map(&tv, v, BHkv, Lk, d) || !make_map(&tdo, dO, BH, Lq, d) ||
      !make_map_f32(&tdqa, ws, BH, Lq, d))
    return ATTN_ERR_CUDA;
  eba::BwdArgs a{};
  a.B = B;
  a.H = H;
  a.group = H / H_kv;
  a.H_kv = H_kv;
  a.Lq = Lq;
  a.Lk = Lk;
  a.n_qtiles = (Lq + eba::kTileRows - 1) / eba::kTileRows;
  a.n_ktiles = (Lk + eba::kTileRows - 1) / eba::kTileRows;
  a.Lq_pad = a.n_qtiles * eba::kTileRows;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq_acc = ws;
  a.nlse2 = ws + BH * Lq * d;
  a.delta = a.nlse2 + BH * a.Lq_pad;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.status = status;
  a.limit_ns = g_wait_limit_ns.load();
  if (static_cast<long long>(a.n_ktiles) * BHkv >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = eba::launch_bwd(tq, tk, tv, tdo, tdqa, a, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H, int d,
                    float scale, void* stream) {
  return attn_fwd_varlen_gqa(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, n_seqs, H, H, d, scale,
                             stream);
}

int attn_fwd_varlen_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H,
                        int H_kv, int d, float scale, void* stream) {
  eba::VarlenTable vt;
  int Tq = 0, Tk = 0;
  int s = build_varlen(cu_seqlens_q, cu_seqlens_k, n_seqs, H, d, scale, false, &vt, &Tq, &Tk);
  if (s != ATTN_OK) return s;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if ((s = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return s;
  int* status = status_word_ptr();
  if (!status) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  if (!make_map_thd(&tq, q, Tq, H, d, false) || !make_map_thd(&tk, k, Tk, H_kv, d, false) ||
      !make_map_thd(&tv, v, Tk, H_kv, d, false))
    return ATTN_ERR_CUDA;
  eba::FwdArgs a{};
  a.B = 1;
  a.H = H;
  a.group = H / H_kv;
  a.Lq = Tq;
  a.Lk = Tk;
  a.n_chunks = 1;
  a.scale_log2 = scale * kLog2e;
  a.o = o;
  a.lse = lse;
  a.status = status;
  a.limit_ns = g_wait_limit_ns.load();
  cudaError_t e = eba::launch_fwd_varlen(tq, tk, tv, a, vt, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

size_t attn_bwd_varlen_workspace_size(int Tq, int H, int d, int n_seqs) {
  if (Tq < 1 || H < 1 || n_seqs < 1 || n_seqs > ATTN_MAX_SEQS || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(Tq) + static_cast<size_t>(eba::kTileRows) * n_seqs;
  return static_cast<size_t>(Tq) * H * d * sizeof(float)  // dQ accumulator
         + 2 * static_cast<size_t>(H) * rows * sizeof(float);  // -lse2 and D
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                    const float* lse, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int n_seqs, int H, int d, float scale,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_varlen_gqa(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, n_seqs,
                             H, H, d, scale, workspace, workspace_bytes, stream);
}

int attn_bwd_varlen_gqa(const void* q, const void* k, const void* v, const void* o,
                        const void* dO, const float* lse, void* dq, void* dk, void* dv,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H,
                        int H_kv, int d, float scale, void* workspace, size_t workspace_bytes,
                        void* stream) {
  eba::VarlenTable vt;
  int Tq = 0, Tk = 0;
  int s = build_varlen(cu_seqlens_q, cu_seqlens_k, n_seqs, H, d, scale, true, &vt, &Tq, &Tk);
  if (s != ATTN_OK) return s;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if ((s = check_ptrs({q, k, v, o, dO, lse, dq, dk, dv})) != ATTN_OK) return s;
  if (!workspace || workspace_bytes < attn_bwd_varlen_workspace_size(Tq, H, d, n_seqs))
    return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  int* status = status_word_ptr();
  if (!status) return ATTN_ERR_CUDA;
  float* ws = static_cast<float*>(workspace);
  CUtensorMap tq, tk, tv, tdo, tdqa;
  if (!make_map_thd(&tq, q, Tq, H, d, false) || !make_map_thd(&tk, k, Tk, H_kv, d, false) ||
      !make_map_thd(&tv, v, Tk, H_kv, d, false) || !make_map_thd(&tdo, dO, Tq, H, d, false) ||
      !make_map_thd(&tdqa, ws, Tq, H, d, true))
    return ATTN_ERR_CUDA;
  eba::BwdArgs a{};
  a.B = 1;
  a.H = H;
  a.group = H / H_kv;
  a.H_kv = H_kv;
  a.Lq = Tq;
  a.Lk = Tk;
  a.Lq_pad = vt.cu_qt[n_seqs] * eba::kTileRows;  // -lse2 / D rows per head
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq_acc = ws;
  a.nlse2 = ws + static_cast<size_t>(Tq) * H * d;
  a.delta = a.nlse2 + static_cast<size_t>(H) * a.Lq_pad;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.status = status;
  a.limit_ns = g_wait_limit_ns.load();
  // Keys of sequences without queries get zero dK, dV (no work item reads
  // them): one fill per run of such sequences, whose rows are contiguous.
  const size_t key_row_bytes = static_cast<size_t>(H_kv) * d * 2;
  for (int s0 = 0; s0 < n_seqs;) {
    if (cu_seqlens_q[s0 + 1] > cu_seqlens_q[s0]) {
      ++s0;
      continue;
    }
    int s1 = s0;
    while (s1 < n_seqs && cu_seqlens_q[s1 + 1] == cu_seqlens_q[s1]) ++s1;
    const size_t off = static_cast<size_t>(cu_seqlens_k[s0]) * key_row_bytes;
    const size_t bytes = static_cast<size_t>(cu_seqlens_k[s1] - cu_seqlens_k[s0]) * key_row_bytes;
    if (bytes > 0) {
      cudaError_t e = cudaMemsetAsync(static_cast<char*>(dk) + off, 0, bytes,
                                      static_cast<cudaStream_t>(stream));
      if (e == cudaSuccess)
        e = cudaMemsetAsync(static_cast<char*>(dv) + off, 0, bytes, static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_fail(e);
    }
    s0 = s1;
  }
  cudaError_t e =
      eba::launch_bwd_varlen(tq, tk, tv, tdo, tdqa, a, vt, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int attn_merge(const float* o_parts, const float* lse_parts, int n_chunks, void* o, float* lse,
               int B, int H, int Lq, int d, void* stream) {
  int s = check_sizes(B, H, Lq, 1, d, 1.0f);
  if (s != ATTN_OK) return s;
  if (n_chunks < 1) return ATTN_ERR_INVALID_ARG;
  if ((s = check_ptrs({o_parts, lse_parts, o, lse})) != ATTN_OK) return s;
  if (bind_device() < 0) return ATTN_ERR_CUDA;
  eba::MergeArgs a{};
  a.o_parts = o_parts;
  a.lse_parts = lse_parts;
  a.n_chunks = n_chunks;
  a.rows = static_cast<long long>(B) * H * Lq;
  a.o = o;
  a.lse = lse;
  cudaError_t e = eba::launch_merge(a, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "an in-kernel wait timed out";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int attn_poll_device_status(void* stream) {
  if (bind_device() < 0) return ATTN_ERR_CUDA;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int value = 0;
  if ((e = cudaMemcpyFromSymbol(&value, g_status_word, sizeof(int))) != cudaSuccess)
    return cuda_fail(e);
  if (value != 0) {
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int))) != cudaSuccess)
      return cuda_fail(e);
  }
  return value == 0 ? ATTN_OK : (value == ATTN_ERR_TIMEOUT ? ATTN_ERR_TIMEOUT : ATTN_ERR_CUDA);
}

int attn_last_cuda_error(void) { return t_last_cuda_error; }

unsigned long long attn_set_wait_limit_ns(unsigned long long ns) {
  constexpr unsigned long long kMaxWaitNs = 1ull << 62;  // kept positive as a signed 64-bit value
  return g_wait_limit_ns.exchange(ns == 0 ? kDefaultWaitNs : (ns > kMaxWaitNs ? kMaxWaitNs : ns));
}

}  // extern "C"
