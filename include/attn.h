/*
 * attn.h - C ABI of the exact blockwise attention library (libattn.so), sm_103a.
 *
 * What the library computes
 * -------------------------
 * Exact softmax attention over long sequences of video tokens, computed block
 * by block with an online softmax so that the Lq x Lk weight matrix is never
 * written to GPU memory:
 *
 *   S = scale * Q K^T,  P = softmax over keys of S,  O = P V,
 *   lse_i = ln sum_j exp(S_ij)                     (natural logarithm)
 *
 * "Training a Large Video Model on a Single Machine in a Day", §3 "Flash
 * Attention" defines attention as a softmax-weighted average of values and
 * adopts the blockwise exact form (§1, §4.1) that keeps memory O(N) in the
 * number of cubified video tokens N. The backward pass recomputes P from the
 * saved lse, keeping only O and lse from the forward pass (activation
 * recomputation, "LV-XAttn", ICML 2025 poster, Abstract). The split-KV pair
 * attn_partial_fwd / attn_merge is the single-GPU form of that poster's
 * cross-attention, where a short query block meets a very long key/value block
 * that stays in place and partial results are merged exactly.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout: Q, O, dO, dQ are [B, H, Lq, d]; K, V, dK, dV are [B, H, Lk, d];
 *    lse is [B, H, Lq]. All contiguous, d fastest. "bf16" arguments point to
 *    __nv_bfloat16 data, "fp32" ones to float.
 *  - Pointers are DEVICE pointers owned by the caller, 16-byte aligned, and
 *    outputs must not overlap inputs or each other.
 *  - Supported head dims: d = 64 or 128. 1 <= B, H; 1 <= Lq, Lk < 2^31;
 *    B * H < 2^31. scale must be finite and > 0 (masked keys are given a
 *    score of -inf before scaling).
 *  - stream is a cudaStream_t (NULL = legacy default stream). Every call is
 *    asynchronous on that stream and returns without waiting for the GPU.
 *    Calls run on the device whose CUDA context is current on the calling
 *    thread (else the CUDA runtime's current device) and may come from any
 *    host thread; a thread without a context gets that device's primary
 *    context bound.
 *  - The library allocates no memory per call. Scratch that a call needs is
 *    passed in by the caller (attn_bwd's workspace).
 *  - Return value: ATTN_OK or an error code. Arguments are validated before
 *    anything is launched, so a call that returns an argument error has no
 *    effect. ATTN_ERR_CUDA means a CUDA launch/attribute call failed;
 *    attn_last_cuda_error then gives the cudaError_t behind it.
 *  - Every wait inside the kernels is bounded (attn_set_wait_limit_ns). A
 *    wait that runs out makes its block stop early and records
 *    ATTN_ERR_TIMEOUT in a per-device status word that
 *    attn_poll_device_status reads; the outputs of that call are then
 *    undefined but the CUDA context stays usable.
 */
#ifndef EBA_ATTN_H
#define EBA_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, range, or scale not finite and > 0 */
  ATTN_ERR_UNSUPPORTED = 2, /* head dim other than 64 / 128, too many chunks */
  ATTN_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  ATTN_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait ran out (from attn_poll_device_status) */
  ATTN_ERR_WORKSPACE = 6    /* workspace missing or smaller than attn_bwd_workspace_size */
};

/* Maximum number of KV chunks accepted by attn_split_fwd. */
#define ATTN_MAX_CHUNKS 64
#define ATTN_MAX_SEQS 1024   /* sequences per packed variable-length call */

/*
 * attn_fwd - forward pass of exact attention.
 *   q [B,H,Lq,d] bf16, k, v [B,H,Lk,d] bf16  (inputs)
 *   o [B,H,Lq,d] bf16, lse [B,H,Lq] fp32      (outputs)
 * O and lse are the values defined at the top of this file. Non-causal: every
 * query attends to every key ("Training a Large Video Model...", §3: video
 * tokens attend jointly over space and time). lse is what attn_bwd needs.
 * Short sequences (Lq and Lk <= 64, e.g. the temporal attention of factorised
 * space-time models) are packed several (batch, head) sequences to a 128-row
 * tile internally, here and in attn_bwd; results and layouts are unchanged.
 * Sequences of 5 to 8 tokens (max(Lq, Lk)) run on the CUDA cores instead,
 * forward and backward, one warp per sequence, with P kept in fp32 (the
 * backward then takes D_i = sum_j P_ij dP_ij and does not read o).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Lq, int Lk, int d, float scale, void* stream);

/*
 * attn_bwd_workspace_size - bytes of scratch attn_bwd needs for these sizes:
 * an fp32 dQ accumulator [B,H,Lq,d] plus two fp32 per-row vectors padded to a
 * multiple of 128 rows (log2-scaled lse and D_i = sum_k dO_ik O_ik). Grows as
 * O(B*H*Lq*d), never with Lq*Lk. Returns 0 for invalid sizes.
 */
size_t attn_bwd_workspace_size(int B, int H, int Lq, int Lk, int d);

/*
 * attn_bwd - gradients of sum(O * dO) with respect to Q, K and V.
 *   q, k, v, o, dO bf16; lse fp32 from attn_fwd (or from attn_merge)
 *   dq [B,H,Lq,d], dk, dv [B,H,Lk,d] bf16 (outputs, fully overwritten)
 *   workspace: device scratch of at least attn_bwd_workspace_size(...) bytes,
 *   16-byte aligned, caller-owned; its contents on entry do not matter.
 * P is recomputed from lse tile by tile (only O and lse are kept from the
 * forward pass), then dV = P^T dO, dP = dO V^T, dS = P * (dP - D),
 * dQ = scale dS K and dK = scale dS^T Q. dQ is accumulated in fp32 with
 * atomic adds, so its low bits may vary from run to run; dK, dV do not.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
             float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fwd_gqa / attn_bwd_gqa - grouped-query attention (the GQA of the
 * MovieGen Llama architecture, NeMo video foundation-model page, "Overview of
 * the video diffusion pipeline"): H query heads share H_kv key/value heads,
 * H a multiple of H_kv; query head h reads K/V head h / (H / H_kv), i.e. each
 * group of H / H_kv consecutive query heads shares one K/V head.
 *   q, o, dO, dq [B, H, Lq, d]; k, v, dk, dv [B, H_kv, Lk, d] bf16; lse
 *   [B, H, Lq] fp32. dK and dV of a K/V head are the sums over its group.
 *   workspace: attn_bwd_workspace_size(B, H, Lq, Lk, d) bytes (query heads).
 *   Everything else as attn_fwd / attn_bwd (H_kv = H is attn_fwd / attn_bwd);
 *   H_kv < 1 or not dividing H: ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int H_kv, int Lq, int Lk, int d, float scale, void* stream);
int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv, int Lq,
                 int Lk, int d, float scale, void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * attn_fwd_fp8 - forward pass with e4m3 (FP8) operands (the FP8 multi-head
 * attention of the NeMo video foundation-model page, "Efficient in-framework
 * inference"), d = 128 only.
 *   q8 [B, H, Lq, 128], k8 [B, H, Lk, 128] and vt8 = V transposed,
 *   [B, H, 128, Lk]: e4m3 (one byte per element), contiguous; the real
 *   values are q8 * q_scale, k8 * k_scale, vt8 * v_scale (per-tensor
 *   dequantisation scales, finite and > 0). Lk must be a multiple of 16 (the
 *   rows of vt8 are TMA-loaded: 16-byte multiples), else ATTN_ERR_MISALIGNED.
 *   o [B, H, Lq, 128] bf16 and lse [B, H, Lq] fp32 as attn_fwd.
 * Scores accumulate in fp32 from the e4m3 products (exact for these inputs);
 * the softmax weights are rounded to e4m3 for the P V product, which is the
 * precision cost of this path (the row sums and lse use the fp32 weights).
 * d != 128: ATTN_ERR_UNSUPPORTED. Other errors as attn_fwd.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, void* o, float* lse, int B,
                 int H, int Lq, int Lk, int d, float scale, float q_scale, float k_scale,
                 float v_scale, void* stream);

/* Size of the scratch buffer built into the library for attn_bwd_noalloc. */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * attn_bwd_noalloc - attn_bwd for callers that cannot allocate device memory.
 * The papers have no counterpart to this entry point; it exists for
 * deployment. Some callers are not allowed to call cudaMalloc: a plugin inside
 * a host application that owns all GPU memory and gives the plugin no
 * allocator, or a serving loop whose memory is fixed at start-up (allocation
 * can synchronise the device and fragment memory, so it is banned after
 * initialisation). They can pass inputs and outputs but not attn_bwd's
 * workspace.
 *   Arguments, layouts and results are those of attn_bwd without the
 *   workspace. The scratch instead comes from one buffer of
 *   ATTN_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library as a static
 *   device array: every GPU that loads the library keeps it reserved until
 *   the process exits.
 *   - Problems with attn_bwd_workspace_size(...) > ATTN_NOALLOC_SCRATCH_BYTES
 *     are refused with ATTN_ERR_WORKSPACE before anything runs (at Lq = 1568,
 *     d = 64, up to B*H = 161 heads fit).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The buffer is reserved on a device by the first call there, not when
 *     the library is loaded (the CUDA runtime loads it lazily): that call
 *     loads it and looks up its device address with the device current. Make
 *     the first call during start-up, before memory runs short and before
 *     any stream capture; a call with B = 0 (other arguments ignored) does
 *     only this set-up and returns ATTN_OK, or ATTN_ERR_CUDA with the CUDA
 *     error kept for attn_last_cuda_error. The address is looked up again
 *     whenever the current context is not the one it was found in (e.g. after
 *     a device reset re-created it).
 *   - Every call shares the buffer of its device and re-initialises what must
 *     start at zero, so consecutive calls on one stream are fine; calls that
 *     overlap on the GPU (concurrent streams) race on it and give wrong
 *     gradients.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk,
                     int d, float scale, void* stream);

/*
 * attn_partial_fwd - attention of every query over the key range [k0, k1) only.
 *   q [B,H,Lq,d], k, v [B,H,Lk,d] bf16 (the full key/value tensors)
 *   o_part [B,H,Lq,d] fp32: the range's own normalised output
 *   lse_part [B,H,Lq] fp32: ln sum over the range of exp(S_ij)
 * 0 <= k0 <= k1 <= Lk. An empty range (k0 == k1) writes o_part = 0 and
 * lse_part = -inf. This is the per-chunk unit of split-KV cross-attention
 * ("LV-XAttn", ICML 2025 poster, Abstract: key/value blocks stay in place).
 */
int attn_partial_fwd(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                     int B, int H, int Lq, int Lk, int d, int k0, int k1, float scale,
                     void* stream);

/*
 * attn_split_fwd - attn_partial_fwd for n_chunks ranges in one launch.
 *   bounds: HOST array of n_chunks + 1 ints, 0 = bounds[0] <= ... <=
 *           bounds[n_chunks] = Lk; chunk c covers keys [bounds[c], bounds[c+1]).
 *   o_parts [n_chunks,B,H,Lq,d] fp32, lse_parts [n_chunks,B,H,Lq] fp32.
 * 1 <= n_chunks <= ATTN_MAX_CHUNKS. Chunk c's outputs equal those of
 * attn_partial_fwd over its range.
 */
int attn_split_fwd(const void* q, const void* k, const void* v, float* o_parts, float* lse_parts,
                   int B, int H, int Lq, int Lk, int d, const int* bounds, int n_chunks,
                   float scale, void* stream);

/*
 * attn_merge - exact merge of n_chunks partial results over disjoint key ranges.
 *   o_parts [n_chunks,B,H,Lq,d] fp32, lse_parts [n_chunks,B,H,Lq] fp32 (inputs)
 *   o [B,H,Lq,d] bf16, lse [B,H,Lq] fp32 (outputs)
 * With M = max_c lse_c: lse = M + ln sum_c exp(lse_c - M) and
 * O = sum_c exp(lse_c - lse) O_c, which equals attention over the union of the
 * ranges ("LV-XAttn", ICML 2025 poster, Lay Summary: the split leaves the
 * model's output unchanged). Chunks with lse_c = -inf carry no weight; a row
 * whose chunks are all empty gets O = 0 and lse = -inf. n_chunks >= 1.
 */
int attn_merge(const float* o_parts, const float* lse_parts, int n_chunks, void* o, float* lse,
               int B, int H, int Lq, int d, void* stream);

/*
 * Packed variable-length sequences ("sequence packing" of the NeMo video
 * foundation-model page: many sequences of different lengths, e.g. image and
 * video token sequences, laid back to back with no padding).
 *
 * Layout is token-major: q, o, dO, dq [Tq, H, d] and k, v, dk, dv [Tk, H, d]
 * bf16, contiguous, d fastest; lse fp32 [H, Tq]. Sequence s owns query tokens
 * [cu_seqlens_q[s], cu_seqlens_q[s+1]) and key/value tokens [cu_seqlens_k[s],
 * cu_seqlens_k[s+1]) and attends only within itself (the exact attention of
 * attn_fwd applied to each sequence). cu_seqlens_q / cu_seqlens_k are HOST
 * arrays of n_seqs + 1 ints: cu[0] = 0, non-decreasing; Tq = cu_seqlens_q[n_seqs],
 * Tk = cu_seqlens_k[n_seqs]; 1 <= n_seqs <= ATTN_MAX_SEQS, Tq, Tk >= 1.
 * Empty sequences are allowed: a sequence with queries but no keys gives
 * O = 0 and lse = -inf for its queries and zero gradients; one without queries
 * gives zero dK, dV for its keys. Other conventions as for attn_fwd/attn_bwd.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H, int d,
                    float scale, void* stream);

/* Packed sequences with grouped-query heads: as attn_fwd_varlen /
 * attn_bwd_varlen, with k, v, dk, dv [Tk, H_kv, d] (H a multiple of H_kv;
 * query head h reads K/V head h / (H / H_kv), as in attn_fwd_gqa). The
 * backward's workspace is attn_bwd_varlen_workspace_size(Tq, H, d, n_seqs).
 * H_kv < 1 or not dividing H: ATTN_ERR_INVALID_ARG. */
int attn_fwd_varlen_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H,
                        int H_kv, int d, float scale, void* stream);
int attn_bwd_varlen_gqa(const void* q, const void* k, const void* v, const void* o,
                        const void* dO, const float* lse, void* dq, void* dk, void* dv,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H,
                        int H_kv, int d, float scale, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Scratch bytes attn_bwd_varlen needs for Tq packed query tokens in at most
 * n_seqs sequences: an fp32 dQ accumulator [Tq, H, d] and two fp32 values per
 * (head, query row) with each sequence padded to whole 128-row tiles (at most
 * Tq + 128 * n_seqs rows). 0 if an argument is invalid. */
size_t attn_bwd_varlen_workspace_size(int Tq, int H, int d, int n_seqs);

/*
 * attn_bwd_varlen - backward pass over packed variable-length sequences.
 * Layout and cu_seqlens as for attn_fwd_varlen; o and lse are that call's
 * outputs. dq is [Tq, H, d], dk, dv [Tk, H, d] bf16. workspace: device memory
 * of at least attn_bwd_varlen_workspace_size(Tq, H, d, n_seqs) bytes, 16-byte
 * aligned, owned by the caller, contents overwritten. Errors as attn_bwd.
 * The dK, dV rows of keys whose sequence has no queries are zeroed by
 * stream-ordered memory fills (one per run of such sequences) before the
 * kernels; every other row is written by the kernels.
 */

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                    const float* lse, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int n_seqs, int H, int d, float scale,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_string(int status);

/*
 * attn_poll_device_status - synchronise `stream`, then read and clear the
 * current device's status word. Returns ATTN_ERR_TIMEOUT if any kernel of this
 * library on this device gave up a bounded wait since the last poll,
 * ATTN_ERR_CUDA if the synchronisation itself failed or a backward kernel found
 * its dynamic shared memory not 1024-byte aligned (it then computed nothing;
 * never observed on GB300), else ATTN_OK.
 */
int attn_poll_device_status(void* stream);

/*
 * attn_last_cuda_error - the error code of the most recent CUDA failure behind
 * an ATTN_ERR_CUDA returned to the calling thread: a cudaError_t, or the
 * CUresult of a failed tensor-map encoding (0 if none yet).
 */
int attn_last_cuda_error(void);

/*
 * attn_set_wait_limit_ns - limit for every in-kernel wait of later launches
 * (process-wide; default 2e9 ns = 2 s). 0 restores the default. Returns the
 * previous value. The waits at a block's teardown, for its own copies and
 * MMAs already in flight, keep a limit of at least 2 s whatever is set here,
 * so even a very short limit only makes blocks stop early (ATTN_ERR_TIMEOUT),
 * never exit with work in flight. Limits above 2^62 ns are stored as 2^62.
 * Time is read from the GPU's global nanosecond timer as a signed difference
 * from the start of each wait: if that timer is stepped back while a wait
 * runs, the wait lasts that much longer instead of ending at once.
 */
unsigned long long attn_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* EBA_ATTN_H */
