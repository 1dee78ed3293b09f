// Fused scaled-dot-product attention forward pass for GB300 (sm_103a).
//
//   O = softmax(scale * Q K^T + mask) V,   LSE = ln sum exp(scale * Q K^T + mask)
//
// The pages behind this kernel (cited by title and section):
//   * "Attention memory" (onecalc.app), sections "The quadratic bound" and
//     "What this memory is": the s x s score matrix between the query-key
//     product and the softmax-weighted sum of values is what naive attention
//     writes to memory.  Section "FlashAttention": walk the keys and values
//     in small blocks, keep running softmax statistics, and never write the
//     s x s matrix.  This kernel keeps each 128 x 128 score tile in tensor
//     memory (TMEM) and never sends it to HBM.
//   * "Flash attention" glossary (news.hamidun.com), second paragraph: tiles
//     that fit on-chip, an incremental numerically stable softmax,
//     parallelism across the sequence (the work units are query tiles), fewer
//     non-matmul operations (exp2 with the scale folded in, packed fp32x2
//     arithmetic, the 1/l division deferred to the epilogue, lazy rescaling
//     of O), and warp specialisation.
//   * "PyTorch attention backends" story (hyper.ai), masked_fill sentences:
//     a masked key scores -inf.  Here the causal and key-padding predicates
//     are evaluated from indices in registers; no mask tensor exists.
//
// Persistent kernel: one CTA per SM walks a static list of work units.  A
// unit is two 128-row query tiles of one (batch, head) against that head's
// allowed keys.  Warp roles (512 threads, four warpgroups):
//   warp 0       TMA producer: per unit the two Q tiles, then K/V tiles into a
//                ring of shared-memory slots guarded by mbarriers.  The ring
//                runs on across units, so the next unit's Q and first K/V
//                tiles load while the current unit finishes.
//   warp 1       tcgen05.mma issuer (one elected lane): S_t = Q_t K_j^T into
//                TMEM, then O_t += P_t V_j with P_t read from TMEM.
//   warps 4-7    softmax for query tile 0; warps 8-11 for query tile 1.  One
//                thread owns one query row (one TMEM lane): it reads its S
//                row, masks, updates the running max and sum, writes P
//                (bf16) back over S, and rescales its O row in TMEM when the
//                max grew by more than 2^8 (lazy correction).
//   warps 12-15  epilogue: O / l rounded to bf16 and written with TMA tensor
//                stores from shared memory, LSE with coalesced stores.
// While one softmax warpgroup works on its tile, the tensor core runs the
// other tile's MMAs, so exp2 work and MMAs overlap; across units, the next
// unit's first steps run while the epilogue warpgroup drains the previous
// O.
//
// Every wait on a barrier is bounded by a %globaltimer deadline.  A wait that
// gives up sets a shared abort flag and a device status word, and every role
// then leaves its loop, waits (bounded) for its own copies and MMAs in
// flight, and the CTA frees its TMEM and exits.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <functional>
#include <mutex>
#include <queue>
#include <type_traits>
#include <utility>
#include <vector>

#include "attn_fwd.h"

namespace {

constexpr int kBM = 128;              // query rows per softmax tile (TMEM lanes)
constexpr int kBN = 128;              // keys per kv tile
constexpr int kQTiles = 2;            // query tiles per work unit
constexpr int kRowsPerUnit = kBM * kQTiles;
constexpr int kListMax = 1024;        // units one CTA may be given by a host-built order
constexpr int kThreads = 384;         // backward kernel: warps 0-3 roles, 4-11 key rows / dQ
constexpr int kFwdThreads = 512;      // forward kernel: warps 0-3 roles, 4-7 / 8-11 softmax, 12-15 epilogue
constexpr int kEpiWarp0 = 12;         // first warp of the forward kernel's epilogue warpgroup
constexpr int kStagePanelBytes = 32 * 128;  // one epilogue warp's O staging: 32 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;   // S0 | S1 | O0 | O1
constexpr int kPanelBytes = 128 * 128;   // one TMA box: 128 rows x 64 bf16 (128 B, swizzled)
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

// Per head dim and element type (kF8: e4m3 Q/K/V and P, else bf16).
template <int D, bool kF8>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!kF8 || D == 128, "e4m3 path: D = 128");
  static constexpr int kEB = kF8 ? 1 : 2;             // bytes per element
  static constexpr int kRowBytes = D * kEB;           // one Q/K/V row
  static constexpr int kPanels = kRowBytes / 128;     // 128-byte swizzle panels per row
  static constexpr int kBoxCols = 128 / kEB;          // elements per TMA box row
  static constexpr int kTileBytes = 128 * kRowBytes;  // one [128 x D] tile
  static constexpr int kQkSteps = kRowBytes / 32;     // MMA K steps of 32 bytes over D
  static constexpr int kKeysPerStep = 32 / kEB;       // keys per P.V MMA K step
  static constexpr int kPvSteps = kBN / kKeysPerStep;
  static constexpr int kPCols = kBN * kEB / 4;        // TMEM columns of packed P
  static constexpr int kOPanels = D / 64;             // 128-byte (64 x bf16) panels of an O row
  // K/V ring depth.  At D = 64 a shallow ring measured best: all CTAs start
  // together and a deep ring makes them all ask DRAM for many tiles at once.
  // At D = 128 four slots leave room for the O staging buffer.
  static constexpr int kSlots = kF8 ? 10 : 4;
  static constexpr bool kTurn = !kF8 && D == 128;  // softmax warpgroups alternate
  static constexpr int kQOff = 0;
  static constexpr int kSlotOff = kQTiles * kTileBytes;
  static constexpr int kStageOff = kSlotOff + kSlots * kTileBytes;  // O staging, 4 KB per epilogue warp
  static constexpr int kStatOff = kStageOff + 4 * kStagePanelBytes;  // float2 (m, l) [kQTiles][kBM]
  static constexpr int kBarOff = kStatOff + kQTiles * kBM * 8;
  // barriers: q_full | q_free[2] | full[kSlots] | empty[kSlots] | s_full[2] | p_full[2] |
  //           o_done[2] | drain | turn | o_free[2] | epi[2] | p_half[2]
  static constexpr int kNumBars = 1 + kQTiles + 2 * kSlots + 3 * kQTiles + 2 + 3 * kQTiles;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // [0] tmem base, [1] abort flag, [2] listed units
  static constexpr int kListOff = kMiscOff + 16;           // uint16 [kListMax]: this CTA's units (host order)
  static constexpr int kSmemBytes = kListOff + 2 * kListMax + 1024;  // + slack for 1024 B alignment
  static constexpr int kOCol0 = kQTiles * kBN;             // first O column in TMEM
  // bf16: the softmax hands P over in two halves of 64 keys, so the first
  // half of P.V runs while the second half's exponentials are computed.
  static constexpr bool kPHalves = !kF8;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct Params {
  uint16_t* o;           // bf16 bits [BH][S_q][D]
  float* lse;            // [BH][S_q]
  const int32_t* kv_valid;
  int S_q;
  int S_kv;
  int H;
  int BH;
  int n_pairs;           // query-tile pairs per (b, h)
  int n_splits;          // key chunks per query pair (1 = no split)
  int n_units;           // BH * n_pairs * n_splits
  float scale_log2;      // scale * log2(e)
  int causal;
  unsigned long long timeout_ns;
  float o_scale;          // multiplies O (the V descale of the e4m3 path, else 1)
  float* o_part;         // split mode: fp32 [n_splits][BH * S_q][D]
  float* lse_part;       // split mode: fp32 [n_splits][BH * S_q]
};

}  // namespace

// Read and cleared by attn_fwd_debug_status.  Bit 0: a bounded wait gave up.
// Bit 1: the backward kernel found its dynamic shared memory off a 1024-byte
// boundary and ran nothing.
__device__ unsigned int g_attn_status = 0;

namespace {

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

struct WaitCtx {
  unsigned long long timeout_ns;
  volatile uint32_t* abort_flag;  // shared memory
};

// Slow path of a bounded wait.  honour_abort=false is used while draining
// work already in flight, which must finish even after another role gave up.
// Inlined: warpgroups with different register budgets (setmaxnreg) cannot
// share one out-of-line function.
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, unsigned long long timeout_ns,
                                            volatile uint32_t* abort_flag, bool honour_abort) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *abort_flag != 0u) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort_flag = 1u;
      atomicOr(&g_attn_status, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, w.timeout_ns, w.abort_flag, true);
}

// The backward kernel has one register budget for the whole CTA, so it keeps
// the slow path out of line (smaller hot loops; measured 2-3% faster there).
__device__ __noinline__ bool mbar_wait_slow_call(uint32_t bar, uint32_t parity, unsigned long long timeout_ns,
                                                 volatile uint32_t* abort_flag, bool honour_abort) {
  return mbar_wait_slow(bar, parity, timeout_ns, abort_flag, honour_abort);
}
__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow_call(bar, parity, w.timeout_ns, w.abort_flag, true);
}
__device__ __forceinline__ bool bwd_wait_drain(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow_call(bar, parity, w.timeout_ns, w.abort_flag, false);
}

// A wait that is expected to last long (a whole work unit): between polls
// the warp sleeps, 64 ns doubling up to 512 ns, so that idle warps leave
// the SM's issue slots and power to the working ones.  Bounded like
// mbar_wait.
__device__ __forceinline__ bool mbar_wait_sleepy(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t ns = 64;
  while (!mbar_try_wait(bar, parity)) {
    if (*w.abort_flag != 0u) return false;
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      *w.abort_flag = 1u;
      atomicOr(&g_attn_status, 1u);
      return false;
    }
    __nanosleep(ns);
    ns = ns < 512u ? 2u * ns : 512u;
  }
  return true;
}

__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, w.timeout_ns, w.abort_flag, false);
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// L2 cache policy for the bulk copies of data read or written once (Q, O):
// those lines go first, so they do not push K and V, which many units
// reread, out of L2.  Measured on GB300 at 4k tokens, 32 heads, causal: DRAM
// reads 122 MB instead of 137 MB (Q + K + V = 101 MB), at the same speed; an
// evict-last policy on the K/V loads changed nothing.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y,
                                                 int z, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(pol)
      : "memory");
}

// Programmatic dependent launch.  The kernel is launched so that it may start
// while the previous kernel in its stream is still finishing: it builds its
// on-chip state (barriers, tensor memory) first and waits here before its
// first global memory access, until that kernel has completed and its writes
// are visible.  Without the launch attribute the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream (if launched the same way) start its own
// prologue on SMs this grid has left; its data accesses still wait for this
// grid to complete.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// shared -> global tensor copy of one box (coordinates of its first element),
// with an L2 cache policy
__device__ __forceinline__ void tma_store_3d_hint(const CUtensorMap* m, uint32_t src, int x, int y, int z,
                                                  uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(x), "r"(y), "r"(z), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's bulk copies have been read
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk copies are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy shared-memory writes become visible to the async proxy (TMA)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4_b32(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Per-warpgroup register budgets of the forward kernel (all four warps of a
// warpgroup execute the same one): the softmax warpgroups take registers the
// others give back.  A launch of kFwdThreads gives every thread
// kRegsAtLaunch; setmaxnreg.dec may only lower that and .inc only raise it
// (anything else is an illegal instruction), so the checks are compile-time.
constexpr uint32_t kRegsAtLaunch = 65536 / kFwdThreads;
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  static_assert(N >= 24 && N % 8 == 0 && N <= kRegsAtLaunch, "setmaxnreg.dec lowers the launch budget");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  static_assert(N <= 256 && N % 8 == 0 && N >= kRegsAtLaunch, "setmaxnreg.inc raises the launch budget");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
// Sets this warpgroup's budget to N: lowers or raises it as N requires.
template <uint32_t N>
__device__ __forceinline__ void regs_set() {
  if constexpr (N < kRegsAtLaunch) regs_dec<N>();
  if constexpr (N > kRegsAtLaunch) regs_inc<N>();
}
// Budgets per warpgroup: warps 0-3 (TMA producer, MMA issuer; more measured
// faster), 4-11 (softmax), 12-15 (epilogue).  With a host-built unit order
// ptxas reports an 8-byte spill at these budgets (a unit index read from
// shared memory cannot be recomputed); 96 / 80 left 4 bytes and measured
// slower, so both instances keep these.
constexpr uint32_t kRegsRoles = 104;
constexpr uint32_t kRegsSoftmax = 168;
constexpr uint32_t kRegsEpi = 72;
static_assert(kRegsRoles + 2 * kRegsSoftmax + kRegsEpi == 4 * kRegsAtLaunch,
              "the budgets share out exactly the launch's registers");

// --- tcgen05 ---------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// One lane of a converged warp (elect.sync); the MMA warp runs warp-wide so
// its addresses and descriptors stay warp-uniform, and only the elected lane
// issues tcgen05.mma / tcgen05.commit.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t e;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(e));
  return e;
}

// Arrive once on `bar` when every tcgen05 op the calling lane issued so far is
// done; only lanes with `pred` set commit.
__device__ __forceinline__ void tc_commit_if(uint32_t pred, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
      "r"(pred)
      : "memory");
}

// D[tmem] (+)= A . B on the tensor core, issued only when `pred` is set (the
// elected lane).  SS: A and B from shared memory; TS: A from tensor memory.
// kind::f16 for bf16 operands, kind::f8f6f4 for e4m3 operands.
template <bool kF8>
__device__ __forceinline__ void mma_ss_if(uint32_t pred, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (kF8) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
        : "memory");
  }
}
template <bool kF8>
__device__ __forceinline__ void mma_ts_if(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (kF8) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
        : "memory");
  }
}

#define ATTN_R32(i) "=r"(r[(i)])
#define ATTN_OUT32                                                                                          \
  ATTN_R32(0), ATTN_R32(1), ATTN_R32(2), ATTN_R32(3), ATTN_R32(4), ATTN_R32(5), ATTN_R32(6), ATTN_R32(7),   \
      ATTN_R32(8), ATTN_R32(9), ATTN_R32(10), ATTN_R32(11), ATTN_R32(12), ATTN_R32(13), ATTN_R32(14),       \
      ATTN_R32(15), ATTN_R32(16), ATTN_R32(17), ATTN_R32(18), ATTN_R32(19), ATTN_R32(20), ATTN_R32(21),     \
      ATTN_R32(22), ATTN_R32(23), ATTN_R32(24), ATTN_R32(25), ATTN_R32(26), ATTN_R32(27), ATTN_R32(28),     \
      ATTN_R32(29), ATTN_R32(30), ATTN_R32(31)
#define ATTN_I32(i) "r"(r[(i)])
#define ATTN_IN32                                                                                           \
  ATTN_I32(0), ATTN_I32(1), ATTN_I32(2), ATTN_I32(3), ATTN_I32(4), ATTN_I32(5), ATTN_I32(6), ATTN_I32(7),   \
      ATTN_I32(8), ATTN_I32(9), ATTN_I32(10), ATTN_I32(11), ATTN_I32(12), ATTN_I32(13), ATTN_I32(14),       \
      ATTN_I32(15), ATTN_I32(16), ATTN_I32(17), ATTN_I32(18), ATTN_I32(19), ATTN_I32(20), ATTN_I32(21),     \
      ATTN_I32(22), ATTN_I32(23), ATTN_I32(24), ATTN_I32(25), ATTN_I32(26), ATTN_I32(27), ATTN_I32(28),     \
      ATTN_I32(29), ATTN_I32(30), ATTN_I32(31)

// 32 consecutive fp32 columns of this thread's TMEM lane -> r[0..31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : ATTN_OUT32
      : "r"(taddr));
}
// r[0..31] -> 32 consecutive columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      ATTN_IN32
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four fp32 -> e4m3 (round to nearest even, saturating), element i in byte i.
__device__ __forceinline__ uint32_t pack_e4m3x4(float p0, float p1, float p2, float p3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(p1), "f"(p0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(p3), "f"(p2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// --- descriptors -----------------------------------------------------------

// Instruction descriptor, fp32 accumulator, M x N.  kind::f16 with bf16 A and
// B (format code 1), or kind::f8f6f4 with e4m3 A and B (format code 0).
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn_major, bool b_mn_major, bool e4m3) {
  return (1u << 4)                                 // D format: f32
         | ((e4m3 ? 0u : 1u) << 7)                 // A format
         | ((e4m3 ? 0u : 1u) << 10)                // B format
         | ((a_mn_major ? 1u : 0u) << 15)          // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)          // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle, K-major operand: rows of
// 128 bytes, 8-row groups 1024 bytes apart (the layout TMA writes).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4)  // start address
         | (static_cast<uint64_t>(1) << 16)             // leading byte offset (unused here)
         | (static_cast<uint64_t>(1024 >> 4) << 32)     // stride byte offset: 8-row group
         | (static_cast<uint64_t>(1) << 46)             // descriptor version (sm_100 family)
         | (static_cast<uint64_t>(2) << 61);            // 128-byte swizzle
}

// Same, MN-major operand (V as the K x N operand with N = head dim
// contiguous): 64-element MN blocks `lbo` bytes apart, 8-row K groups 1024 B.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t addr, uint32_t lbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// S[tmem] = Q_tile[smem] . K_tile[smem]^T over the head dim; every MMA
// consumes 32 bytes of each row (16 bf16 or 32 e4m3 elements).  qd/kd are the
// tiles' base descriptors; a step within a 128-byte swizzle row adds 32 bytes
// (2 in the 16-byte address field), and the next 128-byte panel adds
// kPanelBytes.  Addresses stay below 256 KB, so the 14-bit field never
// carries.
template <int D, bool kF8>
__device__ __forceinline__ void issue_qk(uint32_t pred, uint32_t d_tmem, uint64_t qd, uint64_t kd, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < Cfg<D, kF8>::kQkSteps; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
    mma_ss_if<kF8>(pred, d_tmem, qd + off, kd + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O[tmem] (+)= P[tmem] . V_tile[smem] over the 128 keys; every MMA consumes 32
// bytes of each P row (8 TMEM columns) and kKeysPerStep rows of 128 bytes of
// the MN-major V layout.
template <int D, bool kF8, int kK0 = 0, int kK1 = Cfg<D, kF8>::kPvSteps>
__device__ __forceinline__ void issue_pv(uint32_t pred, uint32_t d_tmem, uint32_t p_tmem, uint64_t vd, uint32_t idesc,
                                         bool accumulate) {
  using C = Cfg<D, kF8>;
#pragma unroll
  for (int kk = kK0; kk < kK1; ++kk) {
    mma_ts_if<kF8>(pred, d_tmem, p_tmem + static_cast<uint32_t>(kk * 8),
                   vd + static_cast<uint64_t>((kk * C::kKeysPerStep * 128) >> 4), idesc,
                   (accumulate || kk > 0) ? 1u : 0u);
  }
}

// --- small arithmetic helpers ----------------------------------------------

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// two fp32 products in one instruction
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// three-input maximum
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// ---------------------------------------------------------------------------
// Work units and shared-memory map
// ---------------------------------------------------------------------------

template <int D, bool kF8>
struct Smem {
  uint32_t base;  // shared address, 1024-aligned
  uint8_t* ptr;   // the same byte as a generic pointer
  __device__ uint32_t q(int t) const { return base + Cfg<D, kF8>::kQOff + t * Cfg<D, kF8>::kTileBytes; }
  __device__ uint32_t stage(int qw) const { return base + Cfg<D, kF8>::kStageOff + qw * kStagePanelBytes; }
  __device__ float2* stat(int t) const { return reinterpret_cast<float2*>(ptr + Cfg<D, kF8>::kStatOff) + t * kBM; }
  __device__ uint32_t slot(int s) const { return base + Cfg<D, kF8>::kSlotOff + s * Cfg<D, kF8>::kTileBytes; }
  __device__ uint32_t bar(int i) const { return base + Cfg<D, kF8>::kBarOff + 8 * i; }
  __device__ uint32_t list() const { return base + Cfg<D, kF8>::kListOff; }
  __device__ int listed() const { return static_cast<int>(reinterpret_cast<const volatile uint32_t*>(ptr + Cfg<D, kF8>::kMiscOff)[2]); }
  __device__ uint32_t bar_q() const { return bar(0); }
  __device__ uint32_t bar_qfree(int t) const { return bar(1 + t); }
  __device__ uint32_t bar_full(int s) const { return bar(1 + kQTiles + s); }
  __device__ uint32_t bar_empty(int s) const { return bar(1 + kQTiles + Cfg<D, kF8>::kSlots + s); }
  __device__ uint32_t bar_s(int t) const { return bar(1 + kQTiles + 2 * Cfg<D, kF8>::kSlots + t); }
  __device__ uint32_t bar_p(int t) const { return bar(1 + 2 * kQTiles + 2 * Cfg<D, kF8>::kSlots + t); }
  __device__ uint32_t bar_o(int t) const { return bar(1 + 3 * kQTiles + 2 * Cfg<D, kF8>::kSlots + t); }
  __device__ uint32_t bar_drain() const { return bar(1 + 4 * kQTiles + 2 * Cfg<D, kF8>::kSlots); }
  __device__ uint32_t bar_turn() const { return bar(2 + 4 * kQTiles + 2 * Cfg<D, kF8>::kSlots); }
  // epilogue warpgroup hand-offs
  __device__ uint32_t bar_ofree(int t) const { return bar(3 + 4 * kQTiles + 2 * Cfg<D, kF8>::kSlots + t); }
  __device__ uint32_t bar_epi(int t) const { return bar(3 + 5 * kQTiles + 2 * Cfg<D, kF8>::kSlots + t); }
  // the first half of P_t (keys 0-63) is in TMEM (kPHalves)
  __device__ uint32_t bar_phalf(int t) const { return bar(3 + 6 * kQTiles + 2 * Cfg<D, kF8>::kSlots + t); }
};

// One work unit: two 128-row query tiles of one (batch, head).
struct Unit {
  int bh;
  int q0;             // first query row
  int nk_pad;         // keys allowed by padding (<= S_kv)
  int split;          // key chunk (0 without splitting)
  int j0;             // first kv tile of the chunk
  int mask_all;       // the chunk lies past every key this unit may see
  int nkv[kQTiles];   // kv tiles each query tile visits from j0 (>= 1)
  int n;              // max over the tiles
};

// Unit u -> coordinates.  Causal: the heaviest query pairs of every head come
// first (longest-processing-time order; long causal launches run these units
// in a host-computed order instead, see build_schedule).  Non-causal: a head's query tiles are
// adjacent, so the CTAs sharing its K/V run side by side and hit in L2.  With
// key splitting, the chunks of one query pair are adjacent units; chunk s of
// a pair whose tiles see at most n kv tiles covers kv tiles
// [s*ceil(n/S), min((s+1)*ceil(n/S), n)).
__device__ __forceinline__ Unit make_unit(const Params& p, int u) {
  Unit w;
  w.split = 0;
  if (p.n_splits > 1) {
    w.split = u % p.n_splits;
    u /= p.n_splits;
  }
  int pair;
  if (p.causal) {
    pair = p.n_pairs - 1 - u / p.BH;
    w.bh = u % p.BH;
  } else {
    w.bh = u / p.n_pairs;
    pair = u % p.n_pairs;
  }
  w.q0 = pair * kRowsPerUnit;
  int nk = p.S_kv;
  if (p.kv_valid != nullptr) nk = min(max(__ldg(p.kv_valid + w.bh / p.H), 0), nk);
  w.nk_pad = nk;
  int tiles[kQTiles];  // kv tiles holding keys each query tile may see
  int n_all = 1;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    const int qs = w.q0 + t * kBM;
    int lim = nk;  // keys any row of this tile may see
    if (qs >= p.S_q) {
      lim = 1;  // tile past the last query row: one kv tile, never stored
    } else if (p.causal) {
      lim = min(lim, min(qs + kBM, p.S_q));
    }
    tiles[t] = (lim + kBN - 1) / kBN;
    n_all = max(n_all, tiles[t]);
  }
  int lo = 0, hi = n_all;
  if (p.n_splits > 1) {
    const int chunk = (n_all + p.n_splits - 1) / p.n_splits;
    lo = w.split * chunk;
    hi = min(lo + chunk, n_all);
  }
  w.mask_all = lo >= hi;  // an empty chunk: one kv tile, every key masked
  if (w.mask_all) {
    lo = 0;
    hi = 1;
  }
  w.j0 = lo;
  w.n = 1;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    // a tile with no keys in the chunk still runs one (fully masked) kv tile
    w.nkv[t] = max(1, min(hi, tiles[t]) - lo);
    w.n = max(w.n, w.nkv[t]);
  }
  return w;
}

// Static snake schedule: in round r, CTA c takes unit r*G + c (r even) or
// r*G + G-1-c (r odd), which evens out the LPT-ordered causal work.
__device__ __forceinline__ int unit_of(int r, int c, int G) { return r * G + ((r & 1) ? (G - 1 - c) : c); }

// Per-CTA unit lists computed on the host (see build_schedule): CTA c runs
// units unit[off[c]] .. unit[off[c + 1] - 1], in that order, each encoded as
// make_unit expects.  Passed by value as a kernel parameter; each CTA copies
// its own list (at most kListMax units) into shared memory before it starts.
constexpr int kTabMaxCtas = 256;
constexpr int kTabMaxUnits = 14336;
struct UnitTable {
  uint16_t off[kTabMaxCtas + 1];
  uint16_t unit[kTabMaxUnits];
};

// The work units of this CTA, in order: with kTab, the list the host built
// (copied into shared memory at kernel start), else the static snake over
// the formula order (which may name units past the end; callers skip those).
__device__ __forceinline__ int ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return static_cast<int>(v);
}

template <bool kTab>
struct UnitSeq {
  uint32_t list;
  int n, G, cta;
  template <int D, bool kF8>
  __device__ UnitSeq(const Params& p, const Smem<D, kF8>& sm)
      : list(sm.list()), G(static_cast<int>(gridDim.x)), cta(static_cast<int>(blockIdx.x)) {
    n = kTab ? sm.listed() : (p.n_units + G - 1) / G;
  }
  __device__ int size() const { return n; }
  __device__ int at(int r) const {
    if constexpr (kTab)
      return ld_shared_u16(list + 2u * static_cast<uint32_t>(r));
    else
      return unit_of(r, cta, G);
  }
};

// ---------------------------------------------------------------------------
// Roles
// ---------------------------------------------------------------------------

// TMA producer (one thread).  Per unit: Q_0, Q_1, then K_0, V_0, K_1, V_1, ...;
// K/V item `it` (counted across units) lives in slot it % kSlots.
template <int D, bool kF8, bool kTab>
__device__ void load_role(const Smem<D, kF8>& sm, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                          const CUtensorMap* tmV, const Params& p, const WaitCtx& w) {
  using C = Cfg<D, kF8>;
  const UnitSeq<kTab> us(p, sm);
  const int rounds = us.size();
  int it = 0;  // K/V items issued
  int k = 0;   // units whose Q was issued
  bool ok = true;
  const uint64_t pol_first = l2_evict_first();  // for Q
  for (int r = 0; r < rounds && ok; ++r) {
    const int u = us.at(r);
    if (u >= p.n_units) continue;
    const Unit un = make_unit(p, u);
    if (k > 0) {  // the previous unit's last S MMAs have read both Q tiles
      ok = mbar_wait(sm.bar_qfree(0), (k - 1) & 1, w) && mbar_wait(sm.bar_qfree(1), (k - 1) & 1, w);
      if (!ok) break;
    }
    mbar_expect_tx(sm.bar_q(), kQTiles * C::kTileBytes);
    for (int t = 0; t < kQTiles; ++t) {
      int y = un.q0 + t * kBM;
      if (y >= p.S_q) y = un.q0;  // a tile wholly past the end reloads tile 0 (never stored)
      for (int pn = 0; pn < C::kPanels; ++pn)
        tma_load_3d_hint(sm.q(t) + pn * kPanelBytes, tmQ, sm.bar_q(), pn * C::kBoxCols, y, un.bh, pol_first);
    }
    ++k;
    for (int j = 0; j < un.n && ok; ++j) {
      for (int kv = 0; kv < 2; ++kv) {
        const int s = it % C::kSlots;
        const int round = it / C::kSlots;
        if (round > 0 && !mbar_wait(sm.bar_empty(s), (round - 1) & 1, w)) {
          ok = false;
          break;
        }
        mbar_expect_tx(sm.bar_full(s), C::kTileBytes);
        const CUtensorMap* m = kv ? tmV : tmK;
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_3d(sm.slot(s) + pn * kPanelBytes, m, sm.bar_full(s), pn * C::kBoxCols, (un.j0 + j) * kBN, un.bh);
        ++it;
      }
    }
  }
  grid_launch_dependents();  // every load of this CTA is issued
  // Every issued copy must land before the CTA can exit (one shared deadline).
  bool drained = (k == 0) || mbar_wait_drain(sm.bar_q(), (k - 1) & 1, w);
  for (int i = (it > C::kSlots ? it - C::kSlots : 0); i < it && drained; ++i)
    drained = mbar_wait_drain(sm.bar_full(i % C::kSlots), (i / C::kSlots) & 1, w);
}

// MMA issuer: the whole warp runs the control flow (so addresses and
// descriptors are warp-uniform); one elected lane issues the MMAs and
// commits.  Per unit and kv step j, for each query tile t that still has
// keys: O_t (+)= P_t V_j, then S_t = Q_t K_{j+1}^T.  P_t is read before the
// next S_t overwrites it because MMAs issued by one thread execute in order.
// Each P_t V waits for P_t (softmax); the first of a unit also waits until
// the epilogue warpgroup has read the previous unit's O_t out of TMEM
// (o_free).
template <int D, bool kF8, bool kTab>
__device__ void mma_role(const Smem<D, kF8>& sm, uint32_t tmem, const Params& p, const WaitCtx& w) {
  using C = Cfg<D, kF8>;
  constexpr uint32_t idesc_s = make_idesc(kBM, kBN, false, false, kF8);
  constexpr uint32_t idesc_pv = make_idesc(kBM, D, false, true, kF8);
  const uint32_t leader = elect_one();
  const uint32_t tS[kQTiles] = {tmem, tmem + kBN};
  const uint32_t tO[kQTiles] = {tmem + C::kOCol0, tmem + C::kOCol0 + D};
  const uint64_t qd[kQTiles] = {sdesc_kmajor_sw128(sm.q(0)), sdesc_kmajor_sw128(sm.q(1))};
  const uint64_t kd0 = sdesc_kmajor_sw128(sm.slot(0));
  const uint64_t vd0 = sdesc_mnmajor_sw128(sm.slot(0), kPanelBytes);
  constexpr uint64_t kSlotStep = C::kTileBytes >> 4;  // descriptor distance between slots
  const UnitSeq<kTab> us(p, sm);
  const int rounds = us.size();
  int it = 0;                // K/V items consumed
  int k = 0;                 // units started
  int pc[kQTiles] = {0, 0};  // P_full phases consumed
  bool ok = true, issued = false;
  for (int r = 0; r < rounds && ok; ++r) {
    const int u = us.at(r);
    if (u >= p.n_units) continue;
    const Unit un = make_unit(p, u);
    const int sk0 = it % C::kSlots;
    ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_q(), k & 1, w) &&
                                     mbar_wait(sm.bar_full(sk0), (it / C::kSlots) & 1, w));
    if (!ok) break;
    tc_fence_after();
#pragma unroll
    for (int t = 0; t < kQTiles; ++t) {  // S_t = Q_t K_0^T (S_t is free: the last P_t V was issued before)
      issue_qk<D, kF8>(leader, tS[t], qd[t], kd0 + sk0 * kSlotStep, idesc_s);
      tc_commit_if(leader, sm.bar_s(t));
      if (un.nkv[t] == 1) tc_commit_if(leader, sm.bar_qfree(t));
    }
    issued = true;
    tc_commit_if(leader, sm.bar_empty(sk0));
    ++it;
    for (int j = 0; j < un.n && ok; ++j) {
      const int iv = it, ik = it + 1;  // V_j, K_{j+1}
      const int sv = iv % C::kSlots, skn = ik % C::kSlots;
      const bool has_next = j + 1 < un.n;
      ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_full(sv), (iv / C::kSlots) & 1, w) &&
                                       (!has_next || mbar_wait(sm.bar_full(skn), (ik / C::kSlots) & 1, w)));
#pragma unroll
      for (int t = 0; t < kQTiles; ++t) {
        if (!ok || j >= un.nkv[t]) continue;
        if constexpr (C::kPHalves) {  // P.V over keys 0-63 as soon as that half of P is in TMEM
          constexpr int kH = C::kPvSteps / 2;
          ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_phalf(t), pc[t] & 1, w));
          if (ok && j == 0 && k > 0) ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_ofree(t), (k - 1) & 1, w));
          if (!ok) continue;
          tc_fence_after();
          issue_pv<D, kF8, 0, kH>(leader, tO[t], tS[t], vd0 + sv * kSlotStep, idesc_pv, j > 0);
          ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_p(t), pc[t] & 1, w));
          ++pc[t];
          if (!ok) continue;
          tc_fence_after();
          issue_pv<D, kF8, kH, C::kPvSteps>(leader, tO[t], tS[t], vd0 + sv * kSlotStep, idesc_pv, true);
        } else {
          ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_p(t), pc[t] & 1, w));
          ++pc[t];
          if (ok && j == 0 && k > 0) ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_ofree(t), (k - 1) & 1, w));
          if (!ok) continue;
          tc_fence_after();
          issue_pv<D, kF8>(leader, tO[t], tS[t], vd0 + sv * kSlotStep, idesc_pv, j > 0);
        }
        tc_commit_if(leader, sm.bar_o(t));
        if (j + 1 < un.nkv[t]) {
          issue_qk<D, kF8>(leader, tS[t], qd[t], kd0 + skn * kSlotStep, idesc_s);
          tc_commit_if(leader, sm.bar_s(t));
          if (j + 2 == un.nkv[t]) tc_commit_if(leader, sm.bar_qfree(t));
        }
      }
      if (!ok) break;
      tc_commit_if(leader, sm.bar_empty(sv));
      ++it;
      if (has_next) {
        tc_commit_if(leader, sm.bar_empty(skn));
        ++it;
      }
    }
    ++k;
  }
  if (issued) {  // all MMAs the leader issued are complete before TMEM is freed
    tc_commit_if(leader, sm.bar_drain());
    __all_sync(0xffffffffu, mbar_wait_drain(sm.bar_drain(), 0, w));
  }
}

// Softmax for query tile t (128 threads, one query row each).  Per kv step it
// reads its S row from TMEM, masks, updates the running max and sum, writes
// P (bf16, or e4m3) back over S and, when the row max grew by more than 2^8,
// rescales O in TMEM before releasing P (lazy correction).  At the end of a
// unit it hands the row's statistics (m, l) to the epilogue warpgroup, which
// normalises and stores O and LSE.
template <int D, bool kSplit, bool kF8, bool kTab>
__device__ void softmax_role(const Smem<D, kF8>& sm, int t, uint32_t tmem, const Params& p, const WaitCtx& w) {
  using C = Cfg<D, kF8>;
  const int r = static_cast<int>(threadIdx.x) - kBM * (1 + t);  // row in tile == TMEM lane
  const int qw = r >> 5;                                         // lane quarter (warp % 4)
  const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
  const uint32_t tS = tmem + lane_off + t * kBN;
  const float c = p.scale_log2;
  const UnitSeq<kTab> us(p, sm);
  const int rounds = us.size();
  int cnt = 0;    // kv tiles this query tile has processed (S_full / O_done phases)
  int sbase = 0;  // softmax steps of both query tiles in this CTA's earlier units
  int k = 0;      // units finished
  bool ok = true;
  for (int rr = 0; rr < rounds && ok; ++rr) {
    const int u = us.at(rr);
    if (u >= p.n_units) continue;
    const Unit un = make_unit(p, u);
    const int qs = un.q0 + t * kBM;
    const int row = qs + r;
    int lim = un.mask_all ? 0 : un.nk_pad;  // keys j < lim are allowed for this row
    if (p.causal) lim = min(lim, row + 1);
    const int nkv = t ? un.nkv[1] : un.nkv[0];
    const int n0 = un.nkv[0], n1 = un.nkv[1];

    float m_c = -INFINITY;  // running max, in scaled log2 units, as used for P
    float l = 0.f;          // running sum of P relative to m_c
    for (int j = 0; j < nkv; ++j) {
      // bf16 at D = 128: the two softmax warpgroups take turns.  The CTA's
      // softmax steps are ordered per unit, per kv step, tile 0 before tile 1,
      // and step n starts its exponentials only once step n - 1 has finished
      // the first half of its own (keys 0-63), so the two warpgroups' bursts
      // of exponentials overlap by half instead of fully, while the tensor
      // core serves the other query tile.  (Measured on GB300: handing the
      // turn over after the first half instead of after both was 3-8% faster
      // at 4k-32k; at D = 64 and with e4m3 operands the MMAs are too short for
      // the alternation to pay, and it costs ~8%.)
      const int step = sbase + min(j, n0) + min(j, n1) + ((t == 1 && j < n0) ? 1 : 0);
      ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_s(t), (cnt + j) & 1, w) &&
                                       (!C::kTurn || step == 0 || mbar_wait(sm.bar_turn(), (step - 1) & 1, w)));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[kBN];
      tmem_ld32(tS + 0, sr + 0);
      tmem_ld32(tS + 32, sr + 32);
      tmem_ld32(tS + 64, sr + 64);
      tmem_ld32(tS + 96, sr + 96);
      tmem_wait_ld();
      float s[kBN];
#pragma unroll
      for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(sr[i]);

      const int kbase = (un.j0 + j) * kBN;
      if (un.mask_all || kbase + kBN > un.nk_pad || (p.causal && kbase + kBN - 1 > qs)) {
        const int lj = lim - kbase;
#pragma unroll
        for (int i = 0; i < kBN; ++i) s[i] = (i < lj) ? s[i] : -INFINITY;
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int i = 0; i < kBN; i += 8) {
        mx0 = max3f(mx0, s[i], s[i + 1]);
        mx1 = max3f(mx1, s[i + 2], s[i + 3]);
        mx2 = max3f(mx2, s[i + 4], s[i + 5]);
        mx3 = max3f(mx3, s[i + 6], s[i + 7]);
      }
      const float new_mc = max3f(mx0, mx1, fmaxf(mx2, mx3)) * c;
      float alpha = 1.f;
      bool rescale_o = false;
      if (new_mc > m_c + kRescaleLog2) {  // also taken on the first tile (m_c = -inf)
        alpha = ex2_approx(m_c - new_mc);
        rescale_o = j > 0;  // O holds data only after the first P.V of the unit
        m_c = new_mc;
      }
      const float mc = (m_c == -INFINITY) ? 0.f : m_c;

      // Lazy correction: O is rescaled only when some row's max grew by > 2^8.
      // (Kept in the softmax warps: every hand-off to a separate warpgroup
      // measured slower than this rarely taken branch.)  It must land before
      // this step's first P.V, which the P hand-off releases.
      auto rescale_if_needed = [&]() {
        if (!__any_sync(0xffffffffu, rescale_o)) return;
        ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_o(t), (cnt + j - 1) & 1, w));
        if (!ok) return;
        tc_fence_after();
        const uint32_t tO = tmem + lane_off + C::kOCol0 + t * D;
        const uint64_t a2 = pack_f32x2(alpha, alpha);
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tO + cc, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float x0, x1;
            unpack_f32x2(mul_f32x2(pack_f32x2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), x0, x1);
            o[i] = __float_as_uint(x0);
            o[i + 1] = __float_as_uint(x1);
          }
          tmem_st32(tO + cc, o);
        }
        tmem_wait_st();
      };

      // p = 2^(s*c - m): one FFMA and one MUFU.EX2 per score; the fp32 p
      // feed the row sum, their packed values feed the P.V MMA.
      uint32_t pk[C::kPCols];
      float sum0 = 0.f, sum1 = 0.f;
      if constexpr (kF8) {  // P as e4m3, four per TMEM column
#pragma unroll
        for (int i = 0; i < kBN / 4; ++i) {
          const float a = ex2_approx(fmaf(s[4 * i], c, -mc));
          const float b = ex2_approx(fmaf(s[4 * i + 1], c, -mc));
          const float e = ex2_approx(fmaf(s[4 * i + 2], c, -mc));
          const float f = ex2_approx(fmaf(s[4 * i + 3], c, -mc));
          sum0 += a + e;
          sum1 += b + f;
          pk[i] = pack_e4m3x4(a, b, e, f);
        }
        l = l * alpha + (sum0 + sum1);  // (this order measured 3-4% faster for e4m3)
#pragma unroll
        for (int cc = 0; cc < C::kPCols; cc += 32) tmem_st32(tS + cc, pk + cc);
        if (C::kTurn) mbar_arrive(sm.bar_turn());
        tmem_wait_st();
        rescale_if_needed();
      } else {  // P as bf16, two per TMEM column, handed over in two halves
        static_assert(C::kPHalves && C::kPCols == 64, "bf16 P: two halves of 32 TMEM columns");
#pragma unroll
        for (int i = 0; i < kBN / 4; ++i) {
          const float a = ex2_approx(fmaf(s[2 * i], c, -mc));
          const float b = ex2_approx(fmaf(s[2 * i + 1], c, -mc));
          sum0 += a;
          sum1 += b;
          pk[i] = pack_bf16x2(a, b);
        }
        tmem_st32(tS, pk);
        if (C::kTurn) mbar_arrive(sm.bar_turn());
        tmem_wait_st();
        rescale_if_needed();
        tc_fence_before();
        mbar_arrive(sm.bar_phalf(t));  // P.V may start on keys 0-63
#pragma unroll
        for (int i = kBN / 4; i < kBN / 2; ++i) {
          const float a = ex2_approx(fmaf(s[2 * i], c, -mc));
          const float b = ex2_approx(fmaf(s[2 * i + 1], c, -mc));
          sum0 += a;
          sum1 += b;
          pk[i] = pack_bf16x2(a, b);
        }
        tmem_st32(tS + 32, pk + 32);
        l = l * alpha + (sum0 + sum1);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(sm.bar_p(t));
    }
    cnt += nkv;
    sbase += n0 + n1;
    if (!ok) break;
    // End of the unit: the row statistics go to the epilogue warpgroup,
    // once it has taken the previous unit's (that epilogue has also read the
    // previous O_t out of TMEM).
    if (k > 0) ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_ofree(t), (k - 1) & 1, w));
    if (!ok) break;
    sm.stat(t)[r] = make_float2(m_c, l);
    mbar_arrive(sm.bar_epi(t));
    ++k;
  }
}

// Epilogue warpgroup (warps 12-15): warp 12 + q serves TMEM lane quarter q
// (rows 32q .. 32q + 31) of both query tiles.  At the end of each unit, tile
// 0 then tile 1, it takes the softmax threads' row statistics (m, l), waits
// for the tile's last P.V, reads O_t out of TMEM (which releases it for the
// next unit's first P.V), scales it by 1/l, rounds to bf16 and writes it
// through a 128-byte-swizzled shared-memory panel with TMA tensor stores
// (one 32-row x 64-column box per panel; rows past S_q are clipped by the
// tensor map).  LSE = (m + log2 l) ln 2 is one coalesced fp32 store per
// row.  With key splitting it writes the fp32 partial O (divided by the
// chunk's own l) and the chunk's LSE to the workspace instead.  Meanwhile
// the softmax warps are already on the next unit's first steps.
template <int D, bool kSplit, bool kF8, bool kTab>
__device__ void epilogue_role(const Smem<D, kF8>& sm, const CUtensorMap* tmO, uint32_t tmem, const Params& p,
                              const WaitCtx& w) {
  using C = Cfg<D, kF8>;
  const int qw = static_cast<int>(threadIdx.x >> 5) & 3;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int rt = qw * 32 + lane;  // row within a query tile == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
  const uint32_t stage = sm.stage(qw);
  const UnitSeq<kTab> us(p, sm);
  const int rounds = us.size();
  int cnt[kQTiles] = {0, 0};  // P.V products of each query tile in earlier units
  int k = 0;                  // units finished
  bool ok = true;
  for (int rr = 0; rr < rounds && ok; ++rr) {
    const int u = us.at(rr);
    if (u >= p.n_units) continue;
    const Unit un = make_unit(p, u);
    // Epilogues of this unit's two query tiles.
#pragma unroll
    for (int t = 0; t < kQTiles; ++t) {
      if (!ok) break;
      const int nkv = un.nkv[t];
      ok = __all_sync(0xffffffffu, mbar_wait_sleepy(sm.bar_epi(t), k & 1, w));
      if (!ok) break;
      const float2 ml = sm.stat(t)[rt];  // (m in scaled log2 units, l)
      ok = __all_sync(0xffffffffu, mbar_wait(sm.bar_o(t), (cnt[t] + nkv - 1) & 1, w));
      cnt[t] += nkv;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tO = tmem + lane_off + C::kOCol0 + t * D;
      const int row0 = un.q0 + t * kBM + qw * 32;  // this warp's first row
      const int row = row0 + lane;
      float inv_l = 0.f, lse = -INFINITY;
      if (ml.y > 0.f) {
        inv_l = p.o_scale / ml.y;  // o_scale: the V descale of the e4m3 path, else 1
        lse = (ml.x + log2f(ml.y)) * kLn2;
      }
      const uint64_t il2 = pack_f32x2(inv_l, inv_l);
      const int64_t grow = static_cast<int64_t>(un.bh) * p.S_q + row;
      if constexpr (kSplit) {  // fp32 partial O of this key chunk, straight from registers
        const int64_t prow = static_cast<int64_t>(un.split) * p.BH * p.S_q + grow;
        float* pdst = p.o_part + prow * D;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tO + cc, o);
          tmem_wait_ld();
          if (row < p.S_q) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float x[4];
#pragma unroll
              for (int e = 0; e < 4; e += 2)
                unpack_f32x2(mul_f32x2(pack_f32x2(__uint_as_float(o[4 * q4 + e]), __uint_as_float(o[4 * q4 + e + 1])),
                                       il2),
                             x[e], x[e + 1]);
              st_global_v4(pdst + cc + 4 * q4, __float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                           __float_as_uint(x[3]));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(sm.bar_ofree(t));
        if (row < p.S_q) p.lse_part[prow] = lse;
      } else {
        // Per 64-column panel: read it out of TMEM (after the last panel O_t
        // is free for the next unit), scale, round to bf16, and write its 32
        // rows x 128 B into the warp's staging panel in the 128-byte swizzle
        // the tensor map expects (16-byte chunk c of row r at chunk position
        // c ^ (r & 7)); then one TMA store.  The next panel is read out of
        // TMEM while the previous store is still reading the staging panel.
        const uint32_t rowa = stage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int pn = 0; pn < C::kOPanels; ++pn) {
          uint32_t pk[32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            tmem_ld32(tO + pn * 64 + h * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              unpack_f32x2(mul_f32x2(pack_f32x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2), x0,
                           x1);
              pk[16 * h + i] = pack_bf16x2(x0, x1);
            }
          }
          if (pn == C::kOPanels - 1) {
            tc_fence_before();
            mbar_arrive(sm.bar_ofree(t));
          }
          if (lane == 0) bulk_wait_read_all();  // the previous store has read the staging panel
          __syncwarp();
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4_b32(rowa + (static_cast<uint32_t>(ch ^ (lane & 7)) << 4), pk[4 * ch], pk[4 * ch + 1],
                             pk[4 * ch + 2], pk[4 * ch + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (row0 < p.S_q) tma_store_3d_hint(tmO, stage, pn * 64, row0, un.bh, l2_evict_first());
            bulk_commit();
          }
        }
        if (row < p.S_q) p.lse[grow] = lse;
      }
    }
    ++k;
  }
  if (lane == 0) bulk_wait_all();  // every O store of this warp is complete before the CTA exits
}

template <int D, bool kSplit, bool kF8, bool kTab>
__device__ __forceinline__ void attn_fwd_body(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                              const CUtensorMap& tmO, const Params& p, const UnitTable* tab) {
  using C = Cfg<D, kF8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const Smem<D, kF8> sm{base, smem};
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);

  if (threadIdx.x == 0) {
    mbar_init(sm.bar_q(), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(sm.bar_full(s), 1);
      mbar_init(sm.bar_empty(s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(sm.bar_qfree(t), 1);
      mbar_init(sm.bar_s(t), 1);
      mbar_init(sm.bar_p(t), kBM);
      mbar_init(sm.bar_o(t), 1);
      mbar_init(sm.bar_ofree(t), kBM);  // the four epilogue warps
      mbar_init(sm.bar_epi(t), kBM);    // the tile's softmax threads
      mbar_init(sm.bar_phalf(t), kBM);  // the tile's softmax threads
    }
    mbar_init(sm.bar_drain(), 1);
    mbar_init(sm.bar_turn(), kBM);
    misc[1] = 0u;
    if (kTab) misc[2] = static_cast<uint32_t>(tab->off[blockIdx.x + 1] - tab->off[blockIdx.x]);
    fence_barrier_init();
  } else if (threadIdx.x == 32) {
    tma_prefetch_desc(&tmQ);  // the tensor maps are kernel parameters, not
    tma_prefetch_desc(&tmK);  // data of the previous kernel
    tma_prefetch_desc(&tmV);
    if (!kSplit) tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(base + C::kMiscOff, kTmemCols);
    tmem_relinquish();
  }
  if (kTab) {  // this CTA's units, from the kernel parameters into shared memory
    const int o0 = tab->off[blockIdx.x], n = tab->off[blockIdx.x + 1] - o0;
    uint16_t* list = reinterpret_cast<uint16_t*>(smem + C::kListOff);
    for (int i = static_cast<int>(threadIdx.x); i < n; i += kFwdThreads) list[i] = tab->unit[o0 + i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtx w{p.timeout_ns, misc + 1};
  // Everything above is on-chip; from here on the kernel reads the previous
  // kernel's outputs (Q, K, V, kv_valid_len) and writes O and LSE.
  grid_dependency_wait();

  // Register budgets per warpgroup: they add up to 4 x 128, the launch's share.
  if (warp < 4) {
    regs_set<kRegsRoles>();
    if (warp == 0) {
      if (lane == 0) load_role<D, kF8, kTab>(sm, &tmQ, &tmK, &tmV, p, w);
    } else if (warp == 1) {
      mma_role<D, kF8, kTab>(sm, tmem, p, w);
    }
  } else if (warp < kEpiWarp0) {
    regs_set<kRegsSoftmax>();
    softmax_role<D, kSplit, kF8, kTab>(sm, (warp - 4) >> 2, tmem, p, w);
  } else {
    regs_set<kRegsEpi>();
    epilogue_role<D, kSplit, kF8, kTab>(sm, &tmO, tmem, p, w);
  }
  grid_launch_dependents();  // this thread has issued all of its work

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The forward kernel: units in the static snake over the formula order.
template <int D, bool kSplit, bool kF8>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_sm103a(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const Params p) {
  attn_fwd_body<D, kSplit, kF8, false>(tmQ, tmK, tmV, tmO, p, nullptr);
}

// The same kernel with each CTA's units listed by the host (long causal
// launches: see build_schedule).
template <int D, bool kF8>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_sm103a_sched(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                          const Params p, const __grid_constant__ UnitTable tab) {
  attn_fwd_body<D, false, kF8, true>(tmQ, tmK, tmV, tmO, p, &tab);
}

// S_kv == 0: every row has no allowed key -> O = 0, LSE = -inf.
__global__ void attn_fill_empty(uint16_t* o, float* lse, int64_t rows, int D) {
  grid_dependency_wait();
  grid_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < rows;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    for (int d = 0; d < D; ++d) o[i * D + d] = 0;
    lse[i] = -INFINITY;
  }
}

// Merge of attention results over disjoint key sets -- the reduction after
// key splitting, and the per-device combine step of ring attention
// ("Flash attention" glossary page, paragraph 4):
//   lse = ln sum_k exp(lse_k),   O = sum_k exp(lse_k - lse) O_k.
// One warp per row; each lane owns D/32 consecutive columns.  Lane j holds
// the weight of part k0 + j of each group of 32 parts and hands it to the
// warp by shuffle; the partial rows are read eight at a time with
// independent loads, so the warp waits for memory once per eight parts, not
// once per part.  A part with lse_k = -inf (no keys) has weight 0; a row
// where every part has -inf gets O = 0 and LSE = -inf.  HBM-bound:
// n_parts * (D + 1) * 4 bytes read and D * 2 + 4 bytes written per row.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const float* __restrict__ o_parts,
                                                         const float* __restrict__ lse_parts, int n_parts,
                                                         int64_t rows, int64_t part_stride_rows,
                                                         uint16_t* __restrict__ o, float* __restrict__ lse) {
  constexpr int kPer = D / 32;  // 4 (float4 per lane) or 2 (float2)
  constexpr int kBatch = 8;     // partial rows in flight per warp
  using Vec = typename std::conditional<kPer == 4, float4, float2>::type;
  grid_dependency_wait();  // the partials come from the kernel before
  grid_launch_dependents();
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int64_t first = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t step = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = first; row < rows; row += step) {
    const float* src = o_parts + row * D + lane * kPer;
    // The first batch of partial rows is requested together with the LSEs,
    // so the two loads overlap instead of following each other.
    Vec v0[kBatch];
    const int n0 = min(kBatch, n_parts);
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (u < n0) v0[u] = __ldg(reinterpret_cast<const Vec*>(src + u * part_stride_rows * D));
    const float lse_mine = lane < n_parts ? __ldg(lse_parts + lane * part_stride_rows + row) : -INFINITY;
    float mx = lse_mine;
    for (int k = lane + 32; k < n_parts; k += 32) mx = fmaxf(mx, __ldg(lse_parts + k * part_stride_rows + row));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float wsum = 0.f;  // this lane's share of the weight sum
    if (mx > -INFINITY) {
      for (int k0 = 0; k0 < n_parts; k0 += 32) {
        const int cnt = min(32, n_parts - k0);
        const float w_mine =
            lane < cnt ? expf((k0 == 0 ? lse_mine : __ldg(lse_parts + (k0 + lane) * part_stride_rows + row)) - mx)
                       : 0.f;
        wsum += w_mine;
        int j = 0;
        if (k0 == 0) {  // the batch already in registers
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            if (u >= n0) break;
            const float wk = __shfl_sync(0xffffffffu, w_mine, u);
            const float* f = reinterpret_cast<const float*>(&v0[u]);
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] += wk * f[e];
          }
          j = n0;
        }
        for (; j + kBatch <= cnt; j += kBatch) {
          Vec v[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u)
            v[u] = __ldg(reinterpret_cast<const Vec*>(src + (k0 + j + u) * part_stride_rows * D));
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const float wk = __shfl_sync(0xffffffffu, w_mine, j + u);
            const float* f = reinterpret_cast<const float*>(&v[u]);
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] += wk * f[e];
          }
        }
        for (; j < cnt; ++j) {
          const Vec v = __ldg(reinterpret_cast<const Vec*>(src + (k0 + j) * part_stride_rows * D));
          const float wk = __shfl_sync(0xffffffffu, w_mine, j);
          const float* f = reinterpret_cast<const float*>(&v);
#pragma unroll
          for (int e = 0; e < kPer; ++e) acc[e] += wk * f[e];
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint32_t packed[kPer / 2];
#pragma unroll
    for (int e = 0; e < kPer / 2; ++e) packed[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    uint16_t* dst = o + row * D + lane * kPer;
    if (kPer == 4)
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[(kPer / 2) - 1]);
    else
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    if (lane == 0) lse[row] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
  }
}

// The backward pass (same anonymous namespace, same PTX wrappers).
#include "attn_bwd.cuh"

// Waits on a barrier nothing completes; the bounded wait must give up.
__global__ void attn_watchdog_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtx w{timeout_ns, &abort_flag};
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, w);
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  });
  return g_encode != nullptr;
}

// [BH][S][D] as a 3-D tensor map with (128 bytes of D) x box_rows x 1 boxes
// and 128-byte swizzle; elements are bf16 (eb = 2), e4m3 bytes (eb = 1) or
// fp32 (eb = 4).  Loads use 128-row boxes; the forward kernel's O stores use
// 32-row boxes (one epilogue warp's rows).
bool encode_3d(CUtensorMap* m, const void* ptr, int D, int S, int64_t BH, int eb = 2, int box_rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * eb, static_cast<cuuint64_t>(S) * D * eb};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = eb == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return g_encode(m, dt, 3,
                  const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Every kernel of the library is launched with programmatic dependent launch:
// it may begin while the previous kernel in the stream is finishing, and
// waits (griddepcontrol.wait) before its first global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 ready, 2 unsupported
std::atomic<int> g_dev_sms[kMaxDevices];

// Checks the device is sm_103, records its SM count and sets the kernels'
// shared-memory limits, once per device.
attn_status_t prepare_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  const int st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st == 1) return ATTN_OK;
  if (st == 2) return ATTN_ERR_UNSUPPORTED;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_DEVICE;
  if (major != 10 || minor != 3) {
    g_dev_state[dev].store(2, std::memory_order_release);
    return ATTN_ERR_UNSUPPORTED;
  }
  if (cudaFuncSetAttribute(attn_fwd_sm103a<64, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<64, false>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_sm103a<128, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128, false>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_sm103a<64, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<64, false>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_sm103a<128, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128, false>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_sm103a<128, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128, true>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_sm103a_sched<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<64, false>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_sm103a_sched<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128, false>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_sm103a_sched<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128, true>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_bwd_sm103a<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<64>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(attn_bwd_sm103a<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<128>::kSmemBytes) != cudaSuccess)
    return ATTN_ERR_DEVICE;
  g_dev_sms[dev].store(std::max(1, sms), std::memory_order_relaxed);
  g_dev_state[dev].store(1, std::memory_order_release);
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Host-computed schedule for long causal launches.  The longest-first order
// balances the CTAs' work but keeps every head's units live at once, at
// different key positions; when the heads' K and V together outgrow L2
// (here: more than kSchedL2Bytes), every unit then streams its keys from
// DRAM (measured at 32k tokens, 32 heads: 11 GB per launch for 1.08 GB of
// inputs and outputs).  Instead, units are taken head by head, heaviest
// query pair first, and the last few heads (whose K and V fit in
// kSchedL2Bytes together) interleaved longest first, so the tail still
// balances; each unit goes to the CTA that is free earliest (greedy list
// scheduling with a unit costing its kv steps plus one).  A handful of heads
// is live at any time.  In simulation at 32k this keeps the balance at
// 0.995 (longest-first: 0.999).
constexpr int64_t kSchedL2Bytes = 64ll << 20;

bool schedule_wanted(int causal, const int32_t* kv_valid_len, int n_splits, int64_t BH, int S_kv, int D, int eb,
                     int n_units, int grid) {
  return causal && kv_valid_len == nullptr && n_splits == 1 && BH * S_kv * static_cast<int64_t>(D) * eb * 2 > kSchedL2Bytes &&
         n_units <= kTabMaxUnits && grid <= kTabMaxCtas;
}

// Returns false (the launch then keeps the formula order) when some CTA would
// be given more than kListMax units.
bool build_schedule(int BH, int n_pairs, int S_q, int S_kv, int D, int eb, int G, UnitTable* tab) {
  const int n_units = BH * n_pairs;
  // kv steps of unit u (encoded as make_unit decodes it when causal)
  auto steps = [&](int u) {
    const int pair = n_pairs - 1 - u / BH;
    int n = 1;
    for (int t = 0; t < kQTiles; ++t) {
      const int qs = pair * kRowsPerUnit + t * kBM;
      const int lim = qs >= S_q ? 1 : std::min(S_kv, std::min(qs + kBM, S_q));
      n = std::max(n, (lim + kBN - 1) / kBN);
    }
    return n;
  };
  const int64_t head_kv = static_cast<int64_t>(S_kv) * D * eb * 2;
  const int k_tail = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(BH, kSchedL2Bytes / head_kv)));
  std::vector<int> order;
  order.reserve(n_units);
  for (int bh = 0; bh < BH - k_tail; ++bh)
    for (int pair = n_pairs - 1; pair >= 0; --pair) order.push_back((n_pairs - 1 - pair) * BH + bh);
  for (int pair = n_pairs - 1; pair >= 0; --pair)
    for (int bh = BH - k_tail; bh < BH; ++bh) order.push_back((n_pairs - 1 - pair) * BH + bh);
  using Slot = std::pair<int64_t, int>;  // (work so far, CTA): the earliest free, lowest index first
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < G; ++c) free_at.push({0, c});
  std::vector<std::vector<uint16_t>> lists(G);
  for (const int u : order) {
    const Slot sl = free_at.top();
    free_at.pop();
    lists[sl.second].push_back(static_cast<uint16_t>(u));
    free_at.push({sl.first + steps(u) + 1, sl.second});
  }
  int pos = 0;
  for (int c = 0; c < G; ++c) {
    if (lists[c].size() > static_cast<size_t>(kListMax)) return false;
    tab->off[c] = static_cast<uint16_t>(pos);
    for (const uint16_t u : lists[c]) tab->unit[pos++] = u;
  }
  tab->off[G] = static_cast<uint16_t>(pos);
  return true;
}

// The last few schedules, by shape (a schedule is a pure function of it).
struct SchedEntry {
  int key[7];
  bool ok;  // build_schedule's result
  UnitTable tab;
};
std::mutex g_sched_mu;
std::vector<SchedEntry> g_sched_cache;

// Copies the schedule for this shape into *out, building and caching it on
// first use; false when the shape has none (see build_schedule).  The copy is
// made under the cache's lock: another thread may evict or move entries as
// soon as it is released.
bool schedule_for(int BH, int n_pairs, int S_q, int S_kv, int D, int eb, int G, UnitTable* out) {
  const int key[7] = {BH, n_pairs, S_q, S_kv, D, eb, G};
  std::lock_guard<std::mutex> lock(g_sched_mu);
  for (const SchedEntry& e : g_sched_cache)
    if (std::equal(key, key + 7, e.key)) {
      if (e.ok) *out = e.tab;
      return e.ok;
    }
  if (g_sched_cache.size() >= 8) g_sched_cache.erase(g_sched_cache.begin());
  g_sched_cache.emplace_back();
  SchedEntry& e = g_sched_cache.back();
  std::copy(key, key + 7, e.key);
  e.ok = build_schedule(BH, n_pairs, S_q, S_kv, D, eb, G, &e.tab);
  if (e.ok) *out = e.tab;
  return e.ok;
}

// Launches the attention kernel; with n_splits > 1 it writes fp32 partials to
// o_part / lse_part instead of o / lse.  kF8: e4m3 Q, K, V; `scale` then
// already includes the Q and K descales and o_scale is the V descale.
template <int D, bool kF8>
attn_status_t launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S_q,
                     int S_kv, float scale, int causal, const int32_t* kv_valid_len, int sms, int n_splits,
                     float* o_part, float* lse_part, cudaStream_t stream, float o_scale = 1.f) {
  using C = Cfg<D, kF8>;
  const int64_t BH = static_cast<int64_t>(B) * H;
  CUtensorMap tq, tk, tv, to;
  if (!encode_3d(&tq, q, D, S_q, BH, C::kEB) || !encode_3d(&tk, k, D, S_kv, BH, C::kEB) ||
      !encode_3d(&tv, v, D, S_kv, BH, C::kEB) || !encode_3d(&to, o, D, S_q, BH, 2, 32))
    return ATTN_ERR_LAUNCH;
  Params prm;
  prm.o = static_cast<uint16_t*>(o);
  prm.lse = lse;
  prm.kv_valid = kv_valid_len;
  prm.S_q = S_q;
  prm.S_kv = S_kv;
  prm.H = H;
  prm.BH = static_cast<int>(BH);
  prm.n_pairs = (S_q + kRowsPerUnit - 1) / kRowsPerUnit;
  prm.n_splits = n_splits;
  prm.n_units = static_cast<int>(BH * prm.n_pairs * n_splits);
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  prm.causal = causal;
  prm.timeout_ns = kDefaultTimeoutNs;
  prm.o_scale = o_scale;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  const int G = std::min(prm.n_units, sms);  // persistent: at most one CTA per SM
  const dim3 grid(static_cast<unsigned>(G));
  cudaError_t e;
  const dim3 block(kFwdThreads);
  UnitTable tab;  // copied into the launch's parameters
  if (schedule_wanted(causal, kv_valid_len, n_splits, BH, S_kv, D, C::kEB, prm.n_units, G) &&
      schedule_for(static_cast<int>(BH), prm.n_pairs, S_q, S_kv, D, C::kEB, G, &tab)) {
    e = launch_pdl(attn_fwd_sm103a_sched<D, kF8>, grid, block, C::kSmemBytes, stream, tq, tk, tv, to, prm, tab);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
  }
  if constexpr (kF8)
    e = launch_pdl(attn_fwd_sm103a<D, false, true>, grid, block, C::kSmemBytes, stream, tq, tk, tv, to, prm);
  else if (n_splits > 1)
    e = launch_pdl(attn_fwd_sm103a<D, true, false>, grid, block, C::kSmemBytes, stream, tq, tk, tv, to, prm);
  else
    e = launch_pdl(attn_fwd_sm103a<D, false, false>, grid, block, C::kSmemBytes, stream, tq, tk, tv, to, prm);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

attn_status_t launch_merge(const float* o_parts, const float* lse_parts, int n_parts, int64_t rows, int D, void* o,
                           float* lse, int sms, cudaStream_t stream) {
  const dim3 blocks(static_cast<unsigned>(std::min<int64_t>((rows + 7) / 8, static_cast<int64_t>(sms) * 16)));
  uint16_t* o16 = static_cast<uint16_t*>(o);
  const cudaError_t e =
      D == 64 ? launch_pdl(attn_merge_kernel<64>, blocks, dim3(256), 0, stream, o_parts, lse_parts, n_parts, rows, rows,
                           o16, lse)
              : launch_pdl(attn_merge_kernel<128>, blocks, dim3(256), 0, stream, o_parts, lse_parts, n_parts, rows, rows,
                           o16, lse);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// Argument checks shared by attn_fwd and attn_fwd_splitkv (nothing is launched).
attn_status_t check_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H,
                         int S_q, int S_kv, int D, float scale, int causal, const int32_t* kv_valid_len) {
  if (B < 1 || H < 1 || S_q < 0 || S_kv < 0) return ATTN_ERR_INVALID_ARG;
  // a buffer may be null only when its extent is zero (empty tensors)
  if (S_q > 0 && (q == nullptr || o == nullptr || lse == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (S_q > 0 && S_kv > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(kv_valid_len, 4))
    return ATTN_ERR_ALIGNMENT;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const int64_t n_pairs = (static_cast<int64_t>(S_q) + kRowsPerUnit - 1) / kRowsPerUnit;
  if (BH * n_pairs > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Backward workspace: lse2 and delta [BH][S_pad] and the fp32 dQ accumulator
// [BH][S_q][D], S_pad = S_q rounded up to whole 128-row tiles.
uint64_t bwd_workspace_bytes(int64_t BH, int64_t S_q, int D) {
  const int64_t S_pad = (S_q + kBM - 1) / kBM * kBM;
  return static_cast<uint64_t>(2 * BH * S_pad + BH * S_q * D) * 4u;
}

template <int D>
attn_status_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* d_o, void* dq, void* dk, void* dv, int B, int H, int S_q, int S_kv, float scale,
                         int causal, const int32_t* kv_valid_len, void* workspace, int sms, cudaStream_t stream) {
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int S_pad = (S_q + kBM - 1) / kBM * kBM;
  float* lse2 = static_cast<float*>(workspace);
  float* delta = lse2 + BH * S_pad;
  float* dq_acc = delta + BH * S_pad;
  const dim3 prep_blocks(static_cast<unsigned>(std::min<int64_t>((BH * S_pad + 7) / 8, static_cast<int64_t>(sms) * 16)));
  if (launch_pdl(attn_bwd_prep<D>, prep_blocks, dim3(256), 0, stream, static_cast<const uint16_t*>(o),
                 static_cast<const uint16_t*>(d_o), lse, lse2, delta, dq_acc, S_q, S_pad, BH) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!encode_3d(&tq, q, D, S_q, BH) || !encode_3d(&tk, k, D, S_kv, BH) || !encode_3d(&tv, v, D, S_kv, BH) ||
      !encode_3d(&tdo, d_o, D, S_q, BH) || !encode_3d(&tdq, dq_acc, D, S_q, BH, 4))
    return ATTN_ERR_LAUNCH;
  BwdParams prm;
  prm.dq_acc = dq_acc;
  prm.lse2 = lse2;
  prm.delta = delta;
  prm.dk = static_cast<uint16_t*>(dk);
  prm.dv = static_cast<uint16_t*>(dv);
  prm.kv_valid = kv_valid_len;
  prm.S_q = S_q;
  prm.S_kv = S_kv;
  prm.S_pad = S_pad;
  prm.H = H;
  prm.BH = static_cast<int>(BH);
  prm.n_kv_tiles = (S_kv + kBN - 1) / kBN;
  prm.n_q_tiles = S_pad / kBM;
  prm.head_group = bwd_head_group(S_q, D);
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  prm.scale = scale;
  prm.causal = causal;
  prm.timeout_ns = kDefaultTimeoutNs;
  const dim3 grid(static_cast<unsigned>(BH * prm.n_kv_tiles));
  if (launch_pdl(attn_bwd_sm103a<D>, grid, dim3(kThreads), BwdCfg<D>::kSmemBytes, stream, tq, tk, tv, tdo, tdq,
                 prm) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  const int64_t n4 = BH * S_q * D / 4;
  const dim3 cv_blocks(static_cast<unsigned>(std::min<int64_t>((n4 + 255) / 256, static_cast<int64_t>(sms) * 16)));
  return launch_pdl(attn_bwd_dq_convert, cv_blocks, dim3(256), 0, stream, static_cast<const float*>(dq_acc),
                    static_cast<uint16_t*>(dq), n4, scale) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_LAUNCH;
}

constexpr int kMaxSplits = 64;

uint64_t splitkv_workspace_bytes(int64_t rows, int D, int n_splits) {
  return static_cast<uint64_t>(n_splits) * static_cast<uint64_t>(rows) * static_cast<uint64_t>(D + 1) * 4u;
}

// Fixed scratch for attn_fwd_splitkv_static: the fp32 partial O and LSE of
// the key chunks live here instead of in a caller-supplied workspace.  It is
// part of the module image, so every device that loads this library holds
// ATTN_STATIC_SCRATCH_BYTES of it until the process exits.  Device code could
// name it directly; host code must ask the runtime for its device address.
static __device__ __align__(256) unsigned char g_static_scratch[ATTN_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void* g_static_addr[kMaxDevices];  // device address of g_static_scratch, per device

// Looks up (once per device, with that device current) where the fixed
// scratch lives on the device.
attn_status_t static_scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_DEVICE;
    g_static_addr[dev] = ptr;
  }
  *out = g_static_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd_abi_version(void) { return 1; }

const char* attn_status_str(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case ATTN_ERR_ALIGNMENT: return "misaligned pointer";
    case ATTN_ERR_LAUNCH: return "kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "in-kernel wait timed out";
    case ATTN_ERR_DEVICE: return "CUDA device error";
  }
  return "unknown status";
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S_q,
                       int S_kv, int D, float scale, int causal, const int32_t* kv_valid_len, void* stream) {
  const attn_status_t as = check_args(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len);
  if (as != ATTN_OK) return as;
  if (S_q == 0) return ATTN_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
  const attn_status_t ps = prepare_device(dev);
  if (ps != ATTN_OK) return ps;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t BH = static_cast<int64_t>(B) * H;

  if (S_kv == 0) {
    const int64_t rows = BH * S_q;
    const dim3 blocks(static_cast<unsigned>(std::min<int64_t>((rows + 255) / 256, 4096)));
    return launch_pdl(attn_fill_empty, blocks, dim3(256), 0, st, static_cast<uint16_t*>(o), lse, rows, D) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_LAUNCH;
  }
  if (!get_encoder()) return ATTN_ERR_DEVICE;
  const int sms = g_dev_sms[dev].load(std::memory_order_relaxed);
  if (D == 64)
    return launch<64, false>(q, k, v, o, lse, B, H, S_q, S_kv, scale, causal, kv_valid_len, sms, 1, nullptr, nullptr, st);
  return launch<128, false>(q, k, v, o, lse, B, H, S_q, S_kv, scale, causal, kv_valid_len, sms, 1, nullptr, nullptr, st);
}

attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                           int S_q, int S_kv, int D, float scale, float q_descale, float k_descale, float v_descale,
                           int causal, const int32_t* kv_valid_len, void* stream) {
  const attn_status_t as = check_args(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len);
  if (as != ATTN_OK) return as;
  if (D != 128) return ATTN_ERR_UNSUPPORTED;
  for (const float d : {q_descale, k_descale, v_descale})
    if (!std::isfinite(d) || !(d > 0.f)) return ATTN_ERR_INVALID_ARG;
  const double s_all = static_cast<double>(scale) * q_descale * k_descale;  // S = s_all * (Q8 . K8)
  if (!(s_all > 0.0) || !std::isfinite(static_cast<float>(s_all)) || static_cast<float>(s_all) == 0.f)
    return ATTN_ERR_INVALID_ARG;
  if (S_q == 0) return ATTN_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
  const attn_status_t ps = prepare_device(dev);
  if (ps != ATTN_OK) return ps;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (S_kv == 0) {
    const int64_t rows = static_cast<int64_t>(B) * H * S_q;
    const dim3 blocks(static_cast<unsigned>(std::min<int64_t>((rows + 255) / 256, 4096)));
    return launch_pdl(attn_fill_empty, blocks, dim3(256), 0, st, static_cast<uint16_t*>(o), lse, rows, D) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_LAUNCH;
  }
  if (!get_encoder()) return ATTN_ERR_DEVICE;
  return launch<128, true>(q, k, v, o, lse, B, H, S_q, S_kv, static_cast<float>(s_all), causal, kv_valid_len,
                           g_dev_sms[dev].load(std::memory_order_relaxed), 1, nullptr, nullptr, st, v_descale);
}

uint64_t attn_bwd_workspace_bytes(int B, int H, int S_q, int D) {
  if (B < 1 || H < 1 || S_q < 0 || (D != 64 && D != 128)) return 0;
  return bwd_workspace_bytes(static_cast<int64_t>(B) * H, S_q, D);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* d_o,
                       void* dq, void* dk, void* dv, int B, int H, int S_q, int S_kv, int D, float scale, int causal,
                       const int32_t* kv_valid_len, void* workspace, uint64_t workspace_bytes, void* stream) {
  const attn_status_t as = check_args(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len);
  if (as != ATTN_OK) return as;
  if (S_q > 0 && (d_o == nullptr || dq == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (S_kv > 0 && (dk == nullptr || dv == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(d_o, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16)) return ATTN_ERR_ALIGNMENT;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH * ((static_cast<int64_t>(S_kv) + kBN - 1) / kBN) > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const uint64_t need = bwd_workspace_bytes(BH, S_q, D);
  if (S_q > 0 && S_kv > 0) {
    if (workspace == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return ATTN_ERR_ALIGNMENT;
    if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  }
  if (S_q == 0 && S_kv == 0) return ATTN_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
  const attn_status_t ps = prepare_device(dev);
  if (ps != ATTN_OK) return ps;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (S_q == 0 || S_kv == 0) {  // no query or no key: every gradient is zero
    const size_t kv_bytes = static_cast<size_t>(BH) * S_kv * D * 2, q_bytes = static_cast<size_t>(BH) * S_q * D * 2;
    if ((kv_bytes && (cudaMemsetAsync(dk, 0, kv_bytes, st) != cudaSuccess ||
                      cudaMemsetAsync(dv, 0, kv_bytes, st) != cudaSuccess)) ||
        (q_bytes && cudaMemsetAsync(dq, 0, q_bytes, st) != cudaSuccess))
      return ATTN_ERR_LAUNCH;
    return ATTN_OK;
  }
  if (!get_encoder()) return ATTN_ERR_DEVICE;
  const int sms = g_dev_sms[dev].load(std::memory_order_relaxed);
  if (D == 64)
    return launch_bwd<64>(q, k, v, o, lse, d_o, dq, dk, dv, B, H, S_q, S_kv, scale, causal, kv_valid_len, workspace,
                          sms, st);
  return launch_bwd<128>(q, k, v, o, lse, d_o, dq, dk, dv, B, H, S_q, S_kv, scale, causal, kv_valid_len, workspace,
                         sms, st);
}

uint64_t attn_fwd_splitkv_workspace_bytes(int B, int H, int S_q, int D, int n_splits) {
  if (B < 1 || H < 1 || S_q < 0 || (D != 64 && D != 128) || n_splits < 1 || n_splits > kMaxSplits) return 0;
  return splitkv_workspace_bytes(static_cast<int64_t>(B) * H * S_q, D, n_splits);
}

int attn_fwd_splitkv_suggest(int B, int H, int S_q, int S_kv, int D, int causal) {
  (void)D;
  (void)causal;
  if (B < 1 || H < 1 || S_q < 1 || S_kv < 1) return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  const int64_t units = static_cast<int64_t>(B) * H * ((S_q + kRowsPerUnit - 1) / kRowsPerUnit);
  if (units >= sms) return 1;
  const int64_t kv_tiles = (S_kv + kBN - 1) / kBN;
  // fill the SMs, but keep at least 4 kv tiles per chunk so a unit's start-up stays small
  const int64_t by_sms = (sms + units - 1) / units;
  const int64_t by_len = std::max<int64_t>(1, kv_tiles / 4);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({by_sms, by_len, kMaxSplits})));
}

int attn_fwd_schedule(int B, int H, int S_q, int S_kv, int D, int elem_bytes, int sms, uint16_t* off,
                      uint16_t* unit, int cap) {
  if (B < 1 || H < 1 || S_q < 1 || S_kv < 1 || (D != 64 && D != 128) || (elem_bytes != 1 && elem_bytes != 2) ||
      sms < 1 || off == nullptr || unit == nullptr)
    return -1;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t n_pairs = (static_cast<int64_t>(S_q) + kRowsPerUnit - 1) / kRowsPerUnit;
  if (BH * n_pairs > INT_MAX) return -1;
  const int n_units = static_cast<int>(BH * n_pairs);
  const int G = std::min(n_units, sms);
  if (!schedule_wanted(1, nullptr, 1, BH, S_kv, D, elem_bytes, n_units, G)) return 0;
  if (cap < n_units) return -1;
  UnitTable tab;
  if (!schedule_for(static_cast<int>(BH), static_cast<int>(n_pairs), S_q, S_kv, D, elem_bytes, G, &tab)) return 0;
  std::copy(tab.off, tab.off + G + 1, off);
  std::copy(tab.unit, tab.unit + n_units, unit);
  return n_units;
}

attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int S_q, int S_kv, int D, float scale, int causal, const int32_t* kv_valid_len,
                               int n_splits, void* workspace, uint64_t workspace_bytes, void* stream) {
  const attn_status_t as = check_args(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len);
  if (as != ATTN_OK) return as;
  if (n_splits < 1 || n_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t rows = BH * S_q;
  if (n_splits > 1) {
    if (workspace == nullptr && rows > 0) return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return ATTN_ERR_ALIGNMENT;
    if (workspace_bytes < splitkv_workspace_bytes(rows, D, n_splits)) return ATTN_ERR_INVALID_ARG;
    if (BH * ((S_q + kRowsPerUnit - 1) / kRowsPerUnit) * n_splits > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  }
  if (n_splits == 1 || S_q == 0 || S_kv == 0)
    return attn_fwd(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len, stream);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
  const attn_status_t ps = prepare_device(dev);
  if (ps != ATTN_OK) return ps;
  if (!get_encoder()) return ATTN_ERR_DEVICE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = g_dev_sms[dev].load(std::memory_order_relaxed);
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = o_part + static_cast<int64_t>(n_splits) * rows * D;
  const attn_status_t ls =
      D == 64 ? launch<64, false>(q, k, v, o, lse, B, H, S_q, S_kv, scale, causal, kv_valid_len, sms, n_splits, o_part,
                           lse_part, st)
              : launch<128, false>(q, k, v, o, lse, B, H, S_q, S_kv, scale, causal, kv_valid_len, sms, n_splits, o_part,
                            lse_part, st);
  if (ls != ATTN_OK) return ls;
  return launch_merge(o_part, lse_part, n_splits, rows, D, o, lse, sms, st);
}

// Key-split forward for callers that cannot allocate device memory: the
// scratch is the fixed array above (see include/attn_fwd.h).  Nothing here
// allocates or frees; a size beyond the fixed scratch is refused before
// anything is launched.
attn_status_t attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                      int S_q, int S_kv, int D, float scale, int causal,
                                      const int32_t* kv_valid_len, int n_splits, void* stream) {
  const attn_status_t as = check_args(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len);
  if (as != ATTN_OK) return as;
  if (n_splits < 1 || n_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(B) * H * S_q;
  if (n_splits > 1 && splitkv_workspace_bytes(rows, D, n_splits) > ATTN_STATIC_SCRATCH_BYTES)
    return ATTN_ERR_UNSUPPORTED;  // the partials would not fit in the fixed scratch
  // Without a split (or with nothing to compute) the scratch is never used:
  // the unsplit path runs without looking up its address.
  if (n_splits == 1 || S_q == 0 || S_kv == 0)
    return attn_fwd(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len, stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
  const attn_status_t ps = prepare_device(dev);
  if (ps != ATTN_OK) return ps;
  void* scratch = nullptr;
  const attn_status_t ss = static_scratch_address(dev, &scratch);
  if (ss != ATTN_OK) return ss;
  return attn_fwd_splitkv(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len, n_splits, scratch,
                          ATTN_STATIC_SCRATCH_BYTES, stream);
}

attn_status_t attn_merge(const float* o_parts, const float* lse_parts, int n_parts, int64_t rows, int D, void* o,
                         float* lse, void* stream) {
  if (n_parts < 1 || n_parts > 4096 || rows < 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return ATTN_OK;
  if (o_parts == nullptr || lse_parts == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
  const attn_status_t ps = prepare_device(dev);
  if (ps != ATTN_OK) return ps;
  return launch_merge(o_parts, lse_parts, n_parts, rows, D, o, lse, g_dev_sms[dev].load(std::memory_order_relaxed),
                      static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_debug_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_DEVICE;
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_attn_status, sizeof word) != cudaSuccess) return ATTN_ERR_DEVICE;
  if (word != 0u && cudaMemcpyToSymbol(g_attn_status, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_DEVICE;
  if (word & 2u) return ATTN_ERR_DEVICE;  // a kernel found its shared memory misaligned and did not run
  return word != 0u ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

attn_status_t attn_watchdog_selftest(uint64_t timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  attn_watchdog_kernel<<<1, 32, 0, st>>>(timeout_ns);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  return attn_fwd_debug_status(stream);
}

}  // extern "C"
