/*
 * attn_fwd.h -- C ABI of the fused scaled-dot-product attention forward pass
 * for NVIDIA GB300 (sm_103a).
 *
 * What is computed (per batch b, head h, query row i):
 *
 *     s_ij   = scale * <q_i, k_j>                  for allowed keys j
 *     O_i    = sum_j softmax_j(s_i.) * v_j
 *     LSE_i  = ln sum_{allowed j} exp(s_ij)
 *
 *   - "Attention memory" page (onecalc.app), sections "The quadratic bound"
 *     and "What this memory is": entry (i, j) of the s x s score matrix is how
 *     much token i attends to token j; it sits between the query-key product
 *     and the softmax-weighted sum of the values.
 *   - Same page, section "FlashAttention", and the "Flash attention" glossary
 *     page (news.hamidun.com), second paragraph: the output is built block by
 *     block over the keys and values with running softmax statistics, so the
 *     s x s matrix is never written to HBM.  The forward calls allocate
 *     nothing; their working set is on-chip (shared memory and tensor
 *     memory).  The library's device image does carry one fixed array of
 *     ATTN_STATIC_SCRATCH_BYTES (32 MiB), the scratch of
 *     attn_fwd_splitkv_static, which every device that loads the library
 *     holds until the process exits.
 *   - "PyTorch attention backends" story (hyper.ai), masked_fill sentences:
 *     a masked key is filled with -inf before the softmax.  Key j is allowed
 *     for row i iff j < S_kv, j < kv_valid_len[b] (when given) and, if causal,
 *     j <= i (top-left alignment, as torch's is_causal).  The mask is never
 *     materialised; it is evaluated from indices inside the kernel.
 *   - A row with no allowed key gets O_i = 0 and LSE_i = -inf.
 *
 * Layout: q, o are bf16 [B][H][S_q][D]; k, v are bf16 [B][H][S_kv][D]; lse is
 * fp32 [B][H][S_q]; all contiguous, row-major.  D is 64 or 128.
 */
#ifndef ATTN_FWD_H_
#define ATTN_FWD_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, scale not finite and > 0 */
  ATTN_ERR_UNSUPPORTED = 2,  /* D not 64/128, device not sm_103, size beyond limits */
  ATTN_ERR_ALIGNMENT = 3,    /* q/k/v/o not 16-byte aligned, lse/kv_valid_len not 4-byte */
  ATTN_ERR_LAUNCH = 4,       /* the CUDA launch (or tensor-map encoding) failed */
  ATTN_ERR_TIMEOUT = 5,      /* a bounded in-kernel wait gave up (see attn_fwd_debug_status) */
  ATTN_ERR_DEVICE = 6        /* CUDA runtime / driver error outside the launch */
} attn_status_t;

/*
 * attn_fwd -- enqueue the attention forward pass on `stream`.
 *
 *   q, k, v       device pointers, bf16, layouts above, 16-byte aligned.
 *   o             device pointer, bf16 [B][H][S_q][D], written.
 *   lse           device pointer, fp32 [B][H][S_q], written (natural log).
 *                 q, o, lse may be NULL when S_q == 0; k, v may be NULL when
 *                 S_kv == 0 (then every row gets O = 0, LSE = -inf).
 *   B, H          >= 1.  S_q, S_kv >= 0 (S_q == 0 is a no-op).
 *   D             64 or 128.
 *   scale         finite and > 0 (usually 1/sqrt(D)).
 *   causal        0 or 1.
 *   kv_valid_len  device int32[B] or NULL (NULL means S_kv for every batch).
 *                 The host never reads it; the kernel clamps each entry to
 *                 [0, S_kv].
 *   stream        a cudaStream_t (NULL = legacy default stream).
 *
 * Asynchronous: returns once the kernel is enqueued.  Every argument check
 * happens before anything is launched; on an error nothing is enqueued and
 * the outputs are untouched.  The caller owns every buffer; the library
 * allocates no device memory.  Thread-safe.  Inputs and outputs must not
 * overlap.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int S_q, int S_kv, int D, float scale, int causal,
                       const int32_t* kv_valid_len, void* stream);

/*
 * attn_fwd_fp8 -- attn_fwd on FP8 (e4m3) inputs, after the FP8 support the
 * "Flash attention" glossary page names for FlashAttention-3 (paragraph 2).
 *
 *   q, k, v       device pointers, e4m3 bytes (1 sign, 4 exponent bits with
 *                 bias 7, 3 mantissa bits), [B][H][S][D], 16-byte aligned.
 *   q_descale, k_descale, v_descale
 *                 per-tensor factors, finite and > 0: the real inputs are
 *                 q_descale * Q8, k_descale * K8, v_descale * V8.
 *   o, lse        as attn_fwd: bf16 O and fp32 natural-log LSE of attention
 *                 over the real (descaled) inputs.
 *   D             128 only (ATTN_ERR_UNSUPPORTED otherwise).
 * S = (scale * q_descale * k_descale) * Q8.K8^T is accumulated exactly in
 * fp32 on the tensor cores (kind::f8f6f4).  The probabilities P enter the
 * P.V product as e4m3 (relative rounding error up to 2^-4 each), while the
 * normaliser l sums them in fp32; O therefore carries a few per cent of
 * relative error and LSE the same accuracy as attn_fwd.  Other arguments,
 * limits and behaviour as attn_fwd.
 */
attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int S_q, int S_kv, int D, float scale, float q_descale,
                           float k_descale, float v_descale, int causal,
                           const int32_t* kv_valid_len, void* stream);

/*
 * attn_bwd -- gradients of attn_fwd's O for a loss with gradient d_o:
 *   P = exp(scale*S - LSE),  dV = P^T dO,  dP = dO V^T,
 *   dS = P * (dP - rowsum(dO * O)),  dQ = scale dS K,  dK = scale dS^T Q,
 * with the same masking as attn_fwd (masked pairs have P = 0).  The "Attention
 * memory" page ("What this memory is") notes that training keeps the s x s
 * scores for this pass unless a fused kernel intervenes; this one recomputes
 * every score tile on chip from Q, K and the forward pass's LSE instead.
 *
 *   q, k, v, o, lse   the inputs and outputs of attn_fwd for the same
 *                     arguments (o bf16 [B][H][S_q][D], lse fp32 [B][H][S_q]).
 *   d_o               device bf16 [B][H][S_q][D], 16-byte aligned.
 *   dq, dk, dv        device bf16, shaped like q, k, v, 16-byte aligned; written.
 *   workspace         caller-owned device buffer, 16-byte aligned, at least
 *                     attn_bwd_workspace_bytes(B, H, S_q, D) bytes (fp32
 *                     per-row statistics and the dQ accumulator); overwritten.
 * D is 64 or 128.  Asynchronous (three kernel launches on `stream`); argument
 * errors are reported before anything is launched.  Key rows that no query
 * may see get dK = dV = 0.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* d_o, void* dq, void* dk, void* dv, int B, int H, int S_q, int S_kv,
                       int D, float scale, int causal, const int32_t* kv_valid_len, void* workspace,
                       uint64_t workspace_bytes, void* stream);

/* Workspace bytes attn_bwd needs (0 for invalid arguments). */
uint64_t attn_bwd_workspace_bytes(int B, int H, int S_q, int D);

/*
 * attn_fwd_splitkv -- the same result as attn_fwd, with the keys of every
 * query tile split into `n_splits` contiguous chunks of whole 128-key tiles
 * that are computed independently (more parallel work when B*H*ceil(S_q/256)
 * is small next to the SM count) and then merged as attn_merge does.
 *   Keys are walked block by block with running softmax statistics ("Flash
 *   attention" glossary page, paragraph 2); combining per-chunk (O, LSE)
 *   pairs by their log-sum-exp is the per-device step of the distributed
 *   ("ring") form of the same tiling (same page, paragraph 4).
 *
 *   n_splits        1 .. 64; 1 calls attn_fwd (workspace unused).
 *   workspace       caller-owned device buffer, 16-byte aligned, at least
 *                   attn_fwd_splitkv_workspace_bytes(B, H, S_q, D, n_splits)
 *                   bytes; holds fp32 partial O [n_splits][B*H*S_q][D] and
 *                   partial LSE [n_splits][B*H*S_q].  Overwritten.
 *   other arguments as attn_fwd.  Asynchronous (two kernel launches); argument
 *   errors are reported before anything is launched.  Calls that share a
 *   workspace must be ordered on one stream.
 */
attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int S_q, int S_kv, int D, float scale, int causal,
                               const int32_t* kv_valid_len, int n_splits, void* workspace,
                               uint64_t workspace_bytes, void* stream);

/* Workspace bytes attn_fwd_splitkv needs (0 for invalid arguments). */
uint64_t attn_fwd_splitkv_workspace_bytes(int B, int H, int S_q, int D, int n_splits);

/*
 * A split count that fills the current device for this shape: 1 when the
 * unsplit work already covers every SM, else enough chunks to do so, with at
 * least 4 kv tiles per chunk (at most 64).
 */
int attn_fwd_splitkv_suggest(int B, int H, int S_q, int S_kv, int D, int causal);

/*
 * attn_fwd_schedule -- the order in which attn_fwd runs the work units of a
 * causal launch of this shape on a device with `sms` SMs, for inspection.
 * Host only: touches no device and launches nothing.
 *
 * A work unit is a pair of 128-row query tiles (256 rows) of one (batch,
 * head): with BH = B*H and n_pairs = ceil(S_q / 256), unit u covers query
 * rows [256 p, 256 p + 256) of head bh = u % BH, where p = n_pairs - 1 -
 * u / BH.  A causal launch without key padding whose K and V together take
 * more than 64 MiB (B*H*S_kv*D*elem_bytes*2 bytes) runs its units in a
 * host-built order: the heads one after another, heaviest query pair first,
 * with the last heads whose K and V fit in 64 MiB interleaved, each unit
 * going to the CTA that is free earliest (greedy list scheduling, a unit
 * costing its kv tiles plus one).  This keeps a few heads' K and V in L2
 * instead of every head's.  Other launches take the units in a fixed
 * longest-first order and have no table.
 *
 *   elem_bytes  2 for bf16 (attn_fwd), 1 for e4m3 (attn_fwd_fp8)
 *   off         host uint16 [min(units, sms) + 1], written: CTA c runs
 *               unit[off[c]] .. unit[off[c + 1] - 1], in that order
 *   unit        host uint16 [cap], written: B*H*n_pairs unit indices
 *
 * Returns the number of units written, 0 when the shape has no host-built
 * order (nothing written), or -1 for an invalid argument (B, H, S_q or S_kv
 * below 1, D not 64 or 128, elem_bytes not 1 or 2, sms below 1, a NULL
 * pointer, more units than fit an int) or a `cap` below the unit count.
 */
int attn_fwd_schedule(int B, int H, int S_q, int S_kv, int D, int elem_bytes, int sms, uint16_t* off,
                      uint16_t* unit, int cap);

/*
 * attn_merge -- combine attention results computed over disjoint key sets:
 *   lse = ln sum_k exp(lse_k),  O = sum_k exp(lse_k - lse) O_k.
 *   o_parts    device fp32 [n_parts][rows][D], 16-byte aligned
 *   lse_parts  device fp32 [n_parts][rows] (natural log; -inf = no keys)
 *   o          device bf16 [rows][D], 16-byte aligned, written
 *   lse        device fp32 [rows], written
 * n_parts 1 .. 4096, D 64 or 128.  A row whose parts are all -inf gets O = 0
 * and LSE = -inf.  Asynchronous.
 */
attn_status_t attn_merge(const float* o_parts, const float* lse_parts, int n_parts, int64_t rows,
                         int D, void* o, float* lse, void* stream);

/*
 * attn_fwd_splitkv_static -- attn_fwd_splitkv without a caller workspace,
 * for callers that cannot allocate device memory: code that runs where every
 * device byte is handed out by some other component's pool and side
 * allocations are not allowed, or where the device-wide synchronisation that
 * cudaMalloc / cudaFree imply cannot be paid at that point.  The pages
 * describe no counterpart; this is a deployment convenience.
 *
 * The partial results live in one fixed array of ATTN_STATIC_SCRATCH_BYTES
 * (32 MiB) that is part of this library's device image; every GPU that loads
 * the library holds it until the process exits.  This call allocates and
 * frees nothing.  It needs n_splits * B*H*S_q * (D + 1) * 4 bytes of that
 * array and returns ATTN_ERR_UNSUPPORTED, launching nothing, when that is
 * more than ATTN_STATIC_SCRATCH_BYTES (use fewer splits, or attn_fwd_splitkv
 * with your own workspace).
 *
 * The first call on each device that splits the keys (n_splits > 1, S_q > 0
 * and S_kv > 0) looks up the array's device address with that device current
 * (cudaGetSymbolAddress) and keeps it; make that first call before any
 * stream capture begins.  Calls that do not split go straight to attn_fwd
 * and never touch the array.
 *
 * The array is shared by every call in the process and keeps whatever the
 * last call left in it; nothing needs to start at zero, because each call
 * writes every partial it later reads.  Calls that can run at the same time on
 * the GPU (different streams, or different host threads without ordering)
 * race on the array: order them on one stream.  Other arguments and the
 * result are as attn_fwd_splitkv.
 */
#define ATTN_STATIC_SCRATCH_BYTES (32ull << 20)
attn_status_t attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int H, int S_q, int S_kv, int D,
                                      float scale, int causal, const int32_t* kv_valid_len,
                                      int n_splits, void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_str(attn_status_t status);

/*
 * attn_fwd_debug_status -- synchronise `stream`, then read and clear the
 * device status word that the kernels set when a bounded wait gives up.
 * Returns ATTN_OK, ATTN_ERR_TIMEOUT, or ATTN_ERR_DEVICE if the
 * synchronisation itself reported a CUDA error or the backward kernel found
 * its dynamic shared memory off a 1024-byte boundary (it then runs nothing).
 */
attn_status_t attn_fwd_debug_status(void* stream);

/*
 * attn_watchdog_selftest -- launch a one-warp kernel that waits on a shared
 * memory barrier nothing ever completes, with the same bounded wait the
 * attention kernel uses and a limit of `timeout_ns` nanoseconds
 * (1e3 .. 1e10).  The kernel gives up, records the timeout and returns; this
 * call then synchronises `stream` and returns what attn_fwd_debug_status
 * returns (ATTN_ERR_TIMEOUT when the watchdog works).  Not part of the
 * attention computation: it exercises the failure path without a GPU fault.
 */
attn_status_t attn_watchdog_selftest(uint64_t timeout_ns, void* stream);

/* Version of this ABI (incremented on incompatible change). */
int attn_fwd_abi_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* ATTN_FWD_H_ */
