// Backward pass of the fused attention, for GB300 (sm_103a).  Included by
// attn_fwd.cu, whose PTX wrappers (TMA, mbarrier, tcgen05) it uses.
//
// Gradients of O = softmax(scale * Q K^T + mask) V for a loss with gradient dO:
//   P   = exp(scale * S - LSE)          (recomputed; LSE from the forward pass)
//   dV  = P^T dO
//   dP  = dO V^T
//   dS  = P * (dP - Delta),  Delta_i = sum_d dO_id O_id  (= sum_j P_ij dP_ij)
//   dQ  = scale * dS K,      dK = scale * dS^T Q
// The training frameworks the "Attention memory" page mentions ("What this
// memory is") keep the s x s scores for this pass unless a fused kernel
// intervenes; here every s x s tile is recomputed on chip from Q, K and the
// per-row LSE, so the backward pass also never holds S or P in HBM.
//
// Kernels:
//   attn_bwd_prep     Delta and LSE*log2(e) per query row (padded to whole
//                     128-row tiles, +inf on padding so P = 0 there), and a
//                     zeroed fp32 dQ accumulator.
//   attn_bwd_sm103a   one CTA per (batch*head, 128-key tile j) walks the query
//                     tiles that see those keys:
//       warp 0        TMA: K_j and V_j once; Q_i into a 2-slot ring and dO_i
//                     into a 1-slot ring.
//       warp 1        tcgen05.mma, warp-wide with one elected issuing lane:
//                       S^T  = K_j Q_i^T            (SS, into TMEM cols [0,128))
//                       dP^T = V_j dO_i^T           (SS, cols [128,256))
//                       dV  += P^T dO_i             (TS: P^T from TMEM)
//                       dK  += dS^T Q_i             (TS: dS^T from TMEM)
//                       dQ_i = dS K_j               (SS: dS from shared memory,
//                                                    into cols [128,128+D))
//       warps 4-7     one key row per thread: P^T and dS^T for the tile
//                     (bf16, back into TMEM and, for dS, into shared memory);
//                     at the end dK and dV out of TMEM into bf16 rows.
//                     At D = 64 warps 8-11 form a second such warpgroup: each
//                     takes 64 of the tile's query columns and half of dQ,
//                     dK and dV (bwd_row_role2), and there is no separate dQ
//                     warpgroup.
//       warps 8-11    one query row per thread: dQ_i out of TMEM into a
//                     shared-memory staging buffer (two boxes of 32 fp32
//                     columns per round), which one thread reduce-adds into
//                     the fp32 accumulator with TMA bulk tensor reductions.
//   attn_bwd_dq_convert  dQ = bf16(scale * accumulator).
// TMEM: S^T | dP^T (then dQ_i) | dV | dK, 512 columns at D = 128.

// (Included inside attn_fwd.cu's anonymous namespace.)

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kPanels = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;  // one [128 x D] bf16 tile
  static constexpr int kQSlots = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;
  static constexpr int kDOOff = kQOff + kQSlots * kTileBytes;
  static constexpr int kDSOff = kDOOff + kTileBytes;           // dS^T [128 keys][128 queries] bf16
  static constexpr int kDSBytes = 128 * 128 * 2;
  static constexpr int kStatOff = kDSOff + kDSBytes;           // [2 tiles][lse2 | delta][128] fp32
  // dQ staging for the TMA reduce-adds: 2 boxes of [128 rows x 32 fp32]
  static constexpr int kStageOff = kStatOff + 2 * 2 * 128 * 4;
  static constexpr int kStageBytes = 2 * 128 * 128;
  static constexpr int kBarOff = kStageOff + kStageBytes;
  // kv_full | q_full[2] | q_empty[2] | do_full | do_empty | s_full | dp_full | p_ready |
  // ds_ready | dq_full | dq_free | dsm_free | done | drain | stat[2] | staged | stage_free |
  // stat2[2] | staged2 | stage_free2 (the second key-row warpgroup)
  static constexpr int kNumBars = 1 + 2 * kQSlots + 2 + 9 + 2 + 2 + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;      // [0] tmem base, [1] abort flag
  // No alignment slack: the kernel checks that the dynamic shared memory
  // starts on a 1024-byte boundary (it does when no static shared memory
  // precedes it) and reports an error instead of running otherwise.
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kStageOff % 1024 == 0, "swizzled staging boxes need 1024-byte alignment");
  static constexpr uint32_t kSCol = 0, kDPCol = 128, kDVCol = 256, kDKCol = 256 + D;
  // D = 64: two key-row warpgroups, each taking 64 of the 128 query columns
  // (and half of the dQ reduction); D = 128: one, plus a dQ warpgroup.
  static constexpr int kRowWGs = (D == 64) ? 2 : 1;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct BwdParams {
  float* dq_acc;            // fp32 [BH][S_q][D], zeroed by attn_bwd_prep
  const float* lse2;        // [BH][S_pad]: LSE * log2(e); +inf for padding and key-less rows
  const float* delta;       // [BH][S_pad]
  uint16_t* dk;             // bf16 [BH][S_kv][D]
  uint16_t* dv;             // bf16 [BH][S_kv][D]
  const int32_t* kv_valid;
  int S_q, S_kv, S_pad, H, BH, n_kv_tiles, n_q_tiles;
  int head_group;           // causal launch order: heads per longest-first group (bwd_head_group)
  float scale_log2;         // scale * log2(e)
  float scale;
  int causal;
  unsigned long long timeout_ns;
};

template <int D>
struct BwdSmem {
  uint32_t base;
  __device__ uint32_t k() const { return base + BwdCfg<D>::kKOff; }
  __device__ uint32_t v() const { return base + BwdCfg<D>::kVOff; }
  __device__ uint32_t q(int s) const { return base + BwdCfg<D>::kQOff + s * BwdCfg<D>::kTileBytes; }
  __device__ uint32_t d_o() const { return base + BwdCfg<D>::kDOOff; }
  __device__ uint32_t ds() const { return base + BwdCfg<D>::kDSOff; }
  __device__ uint32_t bar(int i) const { return base + BwdCfg<D>::kBarOff + 8 * i; }
  __device__ uint32_t kv_full() const { return bar(0); }
  __device__ uint32_t q_full(int s) const { return bar(1 + s); }
  __device__ uint32_t q_empty(int s) const { return bar(3 + s); }
  __device__ uint32_t do_full() const { return bar(5); }
  __device__ uint32_t do_empty() const { return bar(6); }
  __device__ uint32_t s_full() const { return bar(7); }
  __device__ uint32_t dp_full() const { return bar(8); }
  __device__ uint32_t p_ready() const { return bar(9); }
  __device__ uint32_t ds_ready() const { return bar(10); }
  __device__ uint32_t dq_full() const { return bar(11); }
  __device__ uint32_t dq_free() const { return bar(12); }
  __device__ uint32_t dsm_free() const { return bar(13); }
  __device__ uint32_t done() const { return bar(14); }
  __device__ uint32_t drain() const { return bar(15); }
  __device__ uint32_t stat(int b) const { return bar(16 + b); }
  __device__ uint32_t staged() const { return bar(18); }
  __device__ uint32_t stage_free() const { return bar(19); }
  __device__ uint32_t stage() const { return base + BwdCfg<D>::kStageOff; }
  // per key-row warpgroup h (kRowWGs = 2): statistics, staging handshake
  __device__ uint32_t stat_h(int h, int b) const { return h ? bar(20 + b) : stat(b); }
  __device__ uint32_t staged_h(int h) const { return h ? bar(22) : staged(); }
  __device__ uint32_t stage_free_h(int h) const { return h ? bar(23) : stage_free(); }
};

// Heads per longest-first group of the causal launch order (see bwd_work):
// the largest power of two up to 16 whose fp32 dQ accumulators (S_q * D * 4
// bytes per head) take at most 32 MiB, so that they stay in L2 while the
// group's CTAs reduce into them.  Measured on GB300 (causal): at 8k tokens,
// D = 128, groups of 8 moved 631 MB of DRAM traffic instead of 1340 MB with
// 16, at the same speed; at 1k, groups of 4-8 were 6% slower than 16.
inline int bwd_head_group(int S_q, int D) {
  const int64_t head_bytes = static_cast<int64_t>(S_q) * D * 4;
  int g = 16;
  while (g > 1 && g * head_bytes > (32ll << 20)) g >>= 1;
  return g;
}

// What one CTA covers: key tile j of head bh against query tiles
// [i0, i0 + n).  Causal: only query tiles holding a query >= the first key.
struct BwdWork {
  int bh, k0, nk_pad, i0, n;
};

__device__ __forceinline__ BwdWork bwd_work(const BwdParams& p) {
  BwdWork w;
  if (p.causal) {
    // Key tile j walks n - j query tiles.  Heads go in groups of head_group;
    // inside a group the CTAs run longest first (every head's j = 0, then
    // j = 1, ...), so the short CTAs fill the end, while only a group's fp32
    // dQ accumulators are being reduced into at a time and stay in L2.
    const int b = static_cast<int>(blockIdx.x);
    const int g0 = b / (p.head_group * p.n_kv_tiles) * p.head_group;  // first head of the group
    const int gs = min(p.head_group, p.BH - g0);                      // heads in the group
    const int idx = b - g0 * p.n_kv_tiles;
    w.bh = g0 + idx % gs;
    w.k0 = (idx / gs) * kBN;
  } else {  // equal work: a head's key tiles side by side, sharing its Q and dO through L2
    w.bh = static_cast<int>(blockIdx.x) / p.n_kv_tiles;
    w.k0 = (static_cast<int>(blockIdx.x) % p.n_kv_tiles) * kBN;
  }
  int nk = p.S_kv;
  if (p.kv_valid != nullptr) nk = min(max(__ldg(p.kv_valid + w.bh / p.H), 0), nk);
  w.nk_pad = nk;
  w.i0 = p.causal ? min(w.k0 / kBM, p.n_q_tiles) : 0;
  w.n = (w.k0 < nk) ? p.n_q_tiles - w.i0 : 0;  // no valid key in the tile: gradients are zero
  return w;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}


// One key row of P^T for kN query columns of a tile: p = 2^(c s - lse2),
// packed to bf16 pairs.  kMask: column col is allowed iff col >= first.
template <bool kMask, int kN = 128>
__device__ __forceinline__ void bwd_p_row(const uint32_t* sr, const float* st, float c, int first, uint32_t* pk) {
#pragma unroll
  for (int i = 0; i < kN / 4; ++i) {  // four queries at a time
    const float4 l4 = *reinterpret_cast<const float4*>(st + 4 * i);
    const float lse2[4] = {l4.x, l4.y, l4.z, l4.w};
    float pv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x = fmaf(__uint_as_float(sr[4 * i + e]), c, -lse2[e]);
      if (kMask) x = (4 * i + e >= first) ? x : -INFINITY;
      pv[e] = ex2_approx(x);
    }
    pk[2 * i] = pack_bf16x2(pv[0], pv[1]);
    pk[2 * i + 1] = pack_bf16x2(pv[2], pv[3]);
  }
}

// acc[tmem] (+)= A[tmem] . B[smem] over the 128 queries of a tile: the TS
// products dV += P^T dO and dK += dS^T Q.  Every MMA consumes 16 queries (8
// packed TMEM columns of A).  With two key-row warpgroups, the packed columns
// of queries 64-127 start at column 64 (each warpgroup packs in place over its
// own score columns).
template <int D>
__device__ __forceinline__ void bwd_issue_ts(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kBM / 16; ++kk) {
    const uint32_t a_col = (BwdCfg<D>::kRowWGs == 2) ? (kk >> 2) * 64 + (kk & 3) * 8 : kk * 8;
    mma_ts_if<false>(pred, d_tmem, a_tmem + a_col, b_desc + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc,
                     (accumulate || kk > 0) ? 1u : 0u);
  }
}

// TMA producer (one thread).
template <int D>
__device__ void bwd_load_role(const BwdSmem<D>& sm, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                              const CUtensorMap* tmV, const CUtensorMap* tmDO, const BwdWork& wk,
                              const WaitCtx& w) {
  using C = BwdCfg<D>;
  tma_prefetch_desc(tmQ);
  tma_prefetch_desc(tmK);
  tma_prefetch_desc(tmV);
  tma_prefetch_desc(tmDO);
  mbar_expect_tx(sm.kv_full(), 2 * C::kTileBytes);
  for (int pn = 0; pn < C::kPanels; ++pn) {
    tma_load_3d(sm.k() + pn * kPanelBytes, tmK, sm.kv_full(), pn * 64, wk.k0, wk.bh);
    tma_load_3d(sm.v() + pn * kPanelBytes, tmV, sm.kv_full(), pn * 64, wk.k0, wk.bh);
  }
  int nq = 0, ndo = 0;  // Q and dO tiles issued
  for (int t = 0; t < wk.n; ++t) {
    const int y = (wk.i0 + t) * kBM;
    const int qs = t % C::kQSlots;
    if (t >= C::kQSlots && !bwd_wait(sm.q_empty(qs), ((t / C::kQSlots) - 1) & 1, w)) break;
    mbar_expect_tx(sm.q_full(qs), C::kTileBytes);
    for (int pn = 0; pn < C::kPanels; ++pn) tma_load_3d(sm.q(qs) + pn * kPanelBytes, tmQ, sm.q_full(qs), pn * 64, y, wk.bh);
    ++nq;
    if (t > 0 && !bwd_wait(sm.do_empty(), (t - 1) & 1, w)) break;
    mbar_expect_tx(sm.do_full(), C::kTileBytes);
    for (int pn = 0; pn < C::kPanels; ++pn) tma_load_3d(sm.d_o() + pn * kPanelBytes, tmDO, sm.do_full(), pn * 64, y, wk.bh);
    ++ndo;
  }
  // every issued copy lands before the CTA may exit (one shared deadline)
  bool drained = bwd_wait_drain(sm.kv_full(), 0, w);
  for (int u = (nq > C::kQSlots ? nq - C::kQSlots : 0); u < nq && drained; ++u)
    drained = bwd_wait_drain(sm.q_full(u % C::kQSlots), (u / C::kQSlots) & 1, w);
  if (drained && ndo > 0) bwd_wait_drain(sm.do_full(), (ndo - 1) & 1, w);
}

// MMA issuer: warp-wide control flow, one elected lane issues.
template <int D>
__device__ void bwd_mma_role(const BwdSmem<D>& sm, uint32_t tmem, const BwdWork& wk, const WaitCtx& w) {
  using C = BwdCfg<D>;
  constexpr uint32_t idesc_s = make_idesc(kBM, kBN, false, false, false);  // [128 x 128], K-major A and B
  constexpr uint32_t idesc_acc = make_idesc(kBM, D, false, true, false);   // TS: B MN-major
  constexpr uint32_t idesc_dq = make_idesc(kBM, D, true, true, false);     // SS: A and B MN-major
  const uint32_t leader = elect_one();
  const uint64_t kd = sdesc_kmajor_sw128(sm.k());
  const uint64_t vd = sdesc_kmajor_sw128(sm.v());
  const uint64_t k_mn = sdesc_mnmajor_sw128(sm.k(), kPanelBytes);
  const uint64_t ds_mn = sdesc_mnmajor_sw128(sm.ds(), kPanelBytes);
  const uint64_t do_k = sdesc_kmajor_sw128(sm.d_o());
  const uint64_t do_mn = sdesc_mnmajor_sw128(sm.d_o(), kPanelBytes);
  const uint32_t tS = tmem + C::kSCol, tDP = tmem + C::kDPCol, tDV = tmem + C::kDVCol, tDK = tmem + C::kDKCol;
  bool ok = __all_sync(0xffffffffu, bwd_wait(sm.kv_full(), 0, w) && bwd_wait(sm.q_full(0), 0, w));
  bool issued = false;
  if (ok) {
    tc_fence_after();
    issue_qk<D, false>(leader, tS, kd, sdesc_kmajor_sw128(sm.q(0)), idesc_s);  // S^T_0 = K Q_0^T
    tc_commit_if(leader, sm.s_full());
    issued = true;
    ok = __all_sync(0xffffffffu, bwd_wait(sm.do_full(), 0, w));
  }
  if (ok) {
    tc_fence_after();
    issue_qk<D, false>(leader, tDP, vd, do_k, idesc_s);  // dP^T_0 = V dO_0^T
    tc_commit_if(leader, sm.dp_full());
  }
  for (int t = 0; t < wk.n && ok; ++t) {
    const int qs = t % C::kQSlots;
    const uint64_t q_mn = sdesc_mnmajor_sw128(sm.q(qs), kPanelBytes);
    // dV += P^T dO_t  (P^T read from TMEM before S^T_{t+1} overwrites it: in-order MMAs)
    ok = __all_sync(0xffffffffu, bwd_wait(sm.p_ready(), t & 1, w));
    if (!ok) break;
    tc_fence_after();
    bwd_issue_ts<D>(leader, tDV, tS, do_mn, idesc_acc, t > 0);
    tc_commit_if(leader, sm.do_empty());
    if (t + 1 < wk.n) {  // S^T_{t+1}
      const int qn = (t + 1) % C::kQSlots;
      ok = __all_sync(0xffffffffu, bwd_wait(sm.q_full(qn), ((t + 1) / C::kQSlots) & 1, w));
      if (!ok) break;
      tc_fence_after();
      issue_qk<D, false>(leader, tS, kd, sdesc_kmajor_sw128(sm.q(qn)), idesc_s);
      tc_commit_if(leader, sm.s_full());
    }
    // dK += dS^T Q_t (dS^T from TMEM), then dQ_t = dS K into the dP^T columns
    ok = __all_sync(0xffffffffu, bwd_wait(sm.ds_ready(), t & 1, w));
    if (!ok) break;
    tc_fence_after();
    bwd_issue_ts<D>(leader, tDK, tDP, q_mn, idesc_acc, t > 0);
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk) {
      const uint64_t off = static_cast<uint64_t>((kk * 16 * 128) >> 4);
      mma_ss_if<false>(leader, tDP, ds_mn + off, k_mn + off, idesc_dq, kk > 0 ? 1u : 0u);
    }
    tc_commit_if(leader, sm.dq_full());
    tc_commit_if(leader, sm.dsm_free());
    tc_commit_if(leader, sm.q_empty(qs));
    if (t + 1 < wk.n) {  // dP^T_{t+1}, once dQ_t has been read out of its columns
      ok = __all_sync(0xffffffffu, bwd_wait(sm.do_full(), (t + 1) & 1, w) && bwd_wait(sm.dq_free(), t & 1, w));
      if (!ok) break;
      tc_fence_after();
      issue_qk<D, false>(leader, tDP, vd, do_k, idesc_s);
      tc_commit_if(leader, sm.dp_full());
    }
  }
  if (issued) {
    tc_commit_if(leader, sm.done());
    tc_commit_if(leader, sm.drain());
    __all_sync(0xffffffffu, bwd_wait_drain(sm.drain(), 0, w));
  }
}

// Key rows (128 threads): P^T and dS^T per query tile; dK, dV at the end.
template <int D>
__device__ void bwd_row_role(const BwdSmem<D>& sm, uint8_t* smem, uint32_t tmem, const BwdParams& p,
                             const BwdWork& wk, const WaitCtx& w) {
  using C = BwdCfg<D>;
  const int r = static_cast<int>(threadIdx.x) - 128;  // key row == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_off + C::kSCol;
  const uint32_t tDP = tmem + lane_off + C::kDPCol;
  const int key = wk.k0 + r;
  const bool key_ok = key < wk.nk_pad;
  const float c = p.scale_log2;
  float* stats = reinterpret_cast<float*>(smem + C::kStatOff);
  bool ok = true;
  // lse2 and delta of query row r of the next tile, loaded one tile ahead
  const int64_t srow0 = static_cast<int64_t>(wk.bh) * p.S_pad + wk.i0 * kBM + r;
  float next_l2 = 0.f, next_dl = 0.f;
  if (wk.n > 0) {
    next_l2 = __ldg(p.lse2 + srow0);
    next_dl = __ldg(p.delta + srow0);
  }
  for (int t = 0; t < wk.n && ok; ++t) {
    const int q0 = (wk.i0 + t) * kBM;
    // this tile's lse2 and delta, one value per thread into a double buffer;
    // buffer t&1 is rewritten two tiles later, after every thread has passed
    // the next tile's barrier (so it has finished reading this one)
    float* st = stats + (t & 1) * 256;  // [lse2 | delta] of this tile
    st[r] = next_l2;
    st[128 + r] = next_dl;
    if (t + 1 < wk.n) {
      next_l2 = __ldg(p.lse2 + srow0 + (t + 1) * kBM);
      next_dl = __ldg(p.delta + srow0 + (t + 1) * kBM);
    }
    mbar_arrive(sm.stat(t & 1));
    ok = __all_sync(0xffffffffu, bwd_wait(sm.stat(t & 1), (t >> 1) & 1, w));
    if (!ok) break;

    // P^T row: p_c = 2^(c*s_c - lse2_c) for the allowed (key, query) pairs
    ok = __all_sync(0xffffffffu, bwd_wait(sm.s_full(), t & 1, w));
    if (!ok) break;
    tc_fence_after();
    // Masking only on tiles that need it (the causal diagonal, or padded
    // keys): query column col is allowed iff col >= first, and a masked score
    // enters the exponential as -inf, so its P is exactly 0.  Both loops run
    // without a branch per score.  The row is read in two halves of 64
    // columns: a whole row (128 registers) next to the packed P would spill.
    const bool diag = p.causal && q0 < wk.k0 + kBN;  // some query of the tile precedes some key
    const bool masked = diag || wk.k0 + kBN > wk.nk_pad;
    const int first = !key_ok ? kBM : (diag ? key - q0 : 0);
    uint32_t pk[64];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t sr[64];
      tmem_ld32(tS + hh * 64, sr);
      tmem_ld32(tS + hh * 64 + 32, sr + 32);
      tmem_wait_ld();
      if (masked)
        bwd_p_row<true, 64>(sr, st + hh * 64, c, first - hh * 64, pk + hh * 32);
      else
        bwd_p_row<false, 64>(sr, st + hh * 64, c, 0, pk + hh * 32);
    }
    tmem_st32(tS + 0, pk + 0);
    tmem_st32(tS + 32, pk + 32);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(sm.p_ready());

    // dS^T row: p * (dP^T - delta), to TMEM (for dK) and shared memory (for dQ)
    ok = __all_sync(0xffffffffu, bwd_wait(sm.dp_full(), t & 1, w));
    if (ok && t > 0) ok = __all_sync(0xffffffffu, bwd_wait(sm.dsm_free(), (t - 1) & 1, w));
    if (!ok) break;
    tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < 128; cc += 32) {
      uint32_t dpr[32];
      tmem_ld32(tDP + cc, dpr);
      tmem_wait_ld();
      uint32_t dsw[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // four queries at a time
        const float4 d4 = *reinterpret_cast<const float4*>(st + 128 + cc + 4 * i);
        const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t pw = pk[(cc >> 1) + 2 * i + h];
          const float p0 = __uint_as_float(pw << 16), p1 = __uint_as_float(pw & 0xFFFF0000u);
          const float d0 = p0 * (__uint_as_float(dpr[4 * i + 2 * h]) - dl[2 * h]);
          const float d1 = p1 * (__uint_as_float(dpr[4 * i + 2 * h + 1]) - dl[2 * h + 1]);
          dsw[2 * i + h] = pack_bf16x2(d0, d1);
        }
      }
      tmem_st16(tDP + (cc >> 1), dsw);
      // shared memory: row r of the [key][query] tile, 128-byte swizzled panels of 64 queries
      const uint32_t row = sm.ds() + static_cast<uint32_t>((cc >> 6) * kPanelBytes + r * 128);
      const int chunk0 = (cc & 63) >> 3;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_shared_v4_b32(row + static_cast<uint32_t>(((chunk0 + u) ^ (r & 7)) << 4), dsw[4 * u], dsw[4 * u + 1],
                         dsw[4 * u + 2], dsw[4 * u + 3]);
    }
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
    mbar_arrive(sm.ds_ready());
  }

  // dK and dV rows out of TMEM (zero when the CTA had no work)
  bool have = ok && wk.n > 0;
  if (have) have = __all_sync(0xffffffffu, bwd_wait(sm.done(), 0, w));
  if (have) tc_fence_after();
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK (times scale)
    const uint32_t src = tmem + lane_off + (which ? C::kDKCol : C::kDVCol);
    uint16_t* dst = (which ? p.dk : p.dv) + (static_cast<int64_t>(wk.bh) * p.S_kv + key) * D;
    const float f = which ? p.scale : 1.f;
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 32) {
      uint32_t a[32];
      if (have) {
        tmem_ld32(src + cc, a);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = 0u;
      }
      if (key < p.S_kv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wv[e] = pack_bf16x2(__uint_as_float(a[8 * q + 2 * e]) * f, __uint_as_float(a[8 * q + 2 * e + 1]) * f);
          st_global_v4(dst + cc + 8 * q, wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
  }
}

// Query rows (128 threads): dQ_i out of TMEM into shared memory, then TMA
// bulk reduce-adds of the tile into the fp32 accumulator.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int x, int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Key rows with two warpgroups (D = 64): warpgroup hf takes query columns
// [64 hf, 64 hf + 64) of every tile -- P^T and dS^T need no row-wide
// statistic, only LSE and Delta, so the halves never talk to each other --
// and head-dim columns [32 hf, 32 hf + 32) of dQ (one tensor-map box each,
// staged and reduce-added by the warpgroup itself), dK and dV.  dQ_t is read
// out at the start of tile t + 1, before P^T of that tile, so the next dP^T
// product can start while the exponentials run.
template <int D>
__device__ void bwd_row_role2(const BwdSmem<D>& sm, uint8_t* smem, const CUtensorMap* tmDQ, uint32_t tmem,
                              const BwdParams& p, const BwdWork& wk, const WaitCtx& w, int hf) {
  using C = BwdCfg<D>;
  static_assert(C::kRowWGs == 2 && D == 64, "two key-row warpgroups: D = 64");
  constexpr int kN = 64;  // query columns of this warpgroup
  const int r = static_cast<int>(((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31));  // key row == TMEM lane
  const bool leader = (r == 0);
  const uint32_t lane_off = static_cast<uint32_t>(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_off + C::kSCol + hf * kN;    // this half's S^T / P^T columns
  const uint32_t tDP = tmem + lane_off + C::kDPCol + hf * kN;  // this half's dP^T / dS^T columns
  const uint32_t tQ = tmem + lane_off + C::kDPCol + hf * 32;   // dQ_t: row r, this half's 32 head-dim columns
  const int key = wk.k0 + r;
  const bool key_ok = key < wk.nk_pad;
  const float c = p.scale_log2;
  // statistics: [2 tiles][64 lse2 | 64 delta] per warpgroup
  float* stats = reinterpret_cast<float*>(smem + C::kStatOff) + hf * 256;
  const uint32_t box = sm.stage() + static_cast<uint32_t>(hf * kBM * 128);  // this half's dQ staging box
  if (leader) tma_prefetch_desc(tmDQ);
  bool ok = true, issued = false;
  // thread r loads lse2 (r < 64) or delta (r >= 64) of query 64 hf + (r & 63), one tile ahead
  const float* src = (r < 64) ? p.lse2 : p.delta;
  const int64_t srow0 = static_cast<int64_t>(wk.bh) * p.S_pad + wk.i0 * kBM + hf * kN + (r & 63);
  float next_v = (wk.n > 0) ? __ldg(src + srow0) : 0.f;
  int nstaged = 0;
  // dQ of tile tt (this half's columns) out of TMEM, staged, and reduce-added
  auto reduce_dq = [&](int tt) -> bool {
    if (!__all_sync(0xffffffffu, bwd_wait(sm.dq_full(), tt & 1, w))) return false;
    tc_fence_after();
    uint32_t a[32];
    tmem_ld32(tQ, a);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(sm.dq_free());
    if (nstaged > 0) {  // the previous reduction of this box has read it
      if (leader) {
        bulk_wait_read_all();
        mbar_arrive(sm.stage_free_h(hf));
      }
      if (!__all_sync(0xffffffffu, bwd_wait(sm.stage_free_h(hf), (nstaged - 1) & 1, w))) return false;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
      st_shared_v4_b32(box + static_cast<uint32_t>(r * 128 + ((k ^ (r & 7)) << 4)), a[4 * k], a[4 * k + 1],
                       a[4 * k + 2], a[4 * k + 3]);
    fence_async_smem();
    mbar_arrive(sm.staged_h(hf));
    if (leader) {  // rows past the head's last query fall outside the tensor map and are skipped
      if (!bwd_wait(sm.staged_h(hf), nstaged & 1, w)) return false;
      tma_reduce_add_3d(tmDQ, box, 32 * hf, (wk.i0 + tt) * kBM, wk.bh);
      bulk_commit();
      issued = true;
    }
    ++nstaged;
    return true;
  };
  for (int t = 0; t < wk.n && ok; ++t) {
    const int q0 = (wk.i0 + t) * kBM;
    float* st = stats + (t & 1) * 128;  // [lse2 | delta] of this tile's 64 columns
    st[(r < 64 ? 0 : 64) + (r & 63)] = next_v;
    if (t + 1 < wk.n) next_v = __ldg(src + srow0 + (t + 1) * kBM);
    mbar_arrive(sm.stat_h(hf, t & 1));
    ok = __all_sync(0xffffffffu, bwd_wait(sm.stat_h(hf, t & 1), (t >> 1) & 1, w));
    if (!ok) break;
    if (t > 0 && !reduce_dq(t - 1)) {
      ok = false;
      break;
    }

    // P^T row: p_c = 2^(c*s_c - lse2_c) for the allowed (key, query) pairs
    ok = __all_sync(0xffffffffu, bwd_wait(sm.s_full(), t & 1, w));
    if (!ok) break;
    tc_fence_after();
    uint32_t sr[kN];
    tmem_ld32(tS + 0, sr + 0);
    tmem_ld32(tS + 32, sr + 32);
    tmem_wait_ld();
    const int qh = q0 + hf * kN;  // this half's first query
    const bool diag = p.causal && qh < wk.k0 + kBN;
    uint32_t pk[kN / 2];
    if (diag || wk.k0 + kBN > wk.nk_pad) {
      const int first = !key_ok ? kN : (diag ? key - qh : 0);
      bwd_p_row<true, kN>(sr, st, c, first, pk);
    } else {
      bwd_p_row<false, kN>(sr, st, c, 0, pk);
    }
    tmem_st32(tS, pk);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(sm.p_ready());

    // dS^T row: p * (dP^T - delta), to TMEM (for dK) and shared memory (for dQ)
    ok = __all_sync(0xffffffffu, bwd_wait(sm.dp_full(), t & 1, w));
    if (ok && t > 0) ok = __all_sync(0xffffffffu, bwd_wait(sm.dsm_free(), (t - 1) & 1, w));
    if (!ok) break;
    tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < kN; cc += 32) {
      uint32_t dpr[32];
      tmem_ld32(tDP + cc, dpr);
      tmem_wait_ld();
      uint32_t dsw[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // four queries at a time
        const float4 d4 = *reinterpret_cast<const float4*>(st + 64 + cc + 4 * i);
        const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t pw = pk[(cc >> 1) + 2 * i + h];
          const float p0 = __uint_as_float(pw << 16), p1 = __uint_as_float(pw & 0xFFFF0000u);
          const float d0 = p0 * (__uint_as_float(dpr[4 * i + 2 * h]) - dl[2 * h]);
          const float d1 = p1 * (__uint_as_float(dpr[4 * i + 2 * h + 1]) - dl[2 * h + 1]);
          dsw[2 * i + h] = pack_bf16x2(d0, d1);
        }
      }
      tmem_st16(tDP + (cc >> 1), dsw);
      // shared memory: row r of the [key][query] tile, panel hf (queries 64 hf ..), 128-byte swizzle
      const uint32_t row = sm.ds() + static_cast<uint32_t>(hf * kPanelBytes + r * 128);
      const int chunk0 = cc >> 3;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_shared_v4_b32(row + static_cast<uint32_t>(((chunk0 + u) ^ (r & 7)) << 4), dsw[4 * u], dsw[4 * u + 1],
                         dsw[4 * u + 2], dsw[4 * u + 3]);
    }
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
    mbar_arrive(sm.ds_ready());
  }
  if (ok && wk.n > 0) ok = reduce_dq(wk.n - 1);
  if (leader && issued) bulk_wait_all();  // the reductions are complete before the CTA exits

  // this half's head-dim columns of the dK and dV rows (zero when the CTA had no work)
  bool have = ok && wk.n > 0;
  if (have) have = __all_sync(0xffffffffu, bwd_wait(sm.done(), 0, w));
  if (have) tc_fence_after();
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK (times scale)
    const uint32_t srcc = tmem + lane_off + (which ? C::kDKCol : C::kDVCol) + hf * 32;
    uint16_t* dst = (which ? p.dk : p.dv) + (static_cast<int64_t>(wk.bh) * p.S_kv + key) * D + hf * 32;
    const float f = which ? p.scale : 1.f;
    uint32_t a[32];
    if (have) {
      tmem_ld32(srcc, a);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = 0u;
    }
    if (key < p.S_kv) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t wv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          wv[e] = pack_bf16x2(__uint_as_float(a[8 * q + 2 * e]) * f, __uint_as_float(a[8 * q + 2 * e + 1]) * f);
        st_global_v4(dst + 8 * q, wv[0], wv[1], wv[2], wv[3]);
      }
    }
  }
}

template <int D>
__device__ void bwd_dq_role(const BwdSmem<D>& sm, const CUtensorMap* tmDQ, uint32_t tmem, const BwdParams& p,
                            const BwdWork& wk, const WaitCtx& w) {
  using C = BwdCfg<D>;
  const int r = static_cast<int>(threadIdx.x) - 256;  // query row in the tile == TMEM lane
  const bool leader = (r == 0);
  const uint32_t lane_off = static_cast<uint32_t>(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t tQ = tmem + lane_off + C::kDPCol;
  constexpr int kBoxes = D / 32;                  // 32 fp32 (128 B) per box row
  constexpr int kBoxBytes = kBM * 128;            // one [128 rows x 32 fp32] box
  if (leader) tma_prefetch_desc(tmDQ);
  bool issued = false;
  int nround = 0;  // staging rounds so far
  for (int t = 0; t < wk.n; ++t) {
    if (!__all_sync(0xffffffffu, bwd_wait(sm.dq_full(), t & 1, w))) break;
    tc_fence_after();
    // read the whole row first and release its TMEM columns (the next dP^T
    // product waits for them)
    uint32_t a[D];
#pragma unroll
    for (int cc = 0; cc < D; cc += 32) tmem_ld32(tQ + cc, a + cc);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(sm.dq_free());
    // Stage row r in the layout of the accumulator's tensor-map boxes (box c:
    // head-dim columns [32c, 32c + 32) of the 128 rows, 128 B per row, 16-byte
    // chunks XOR-swizzled by row & 7, which also puts the 32 rows a warp
    // writes at once in different banks), two boxes per round through the
    // staging buffer; the leader reduce-adds each round into the accumulator
    // and frees the buffer once the TMA has read it.
    const int q0 = (wk.i0 + t) * kBM;
    bool ok = true;
#pragma unroll
    for (int rd = 0; rd < kBoxes / 2; ++rd) {
      ok = __all_sync(0xffffffffu, nround == 0 || bwd_wait(sm.stage_free(), (nround - 1) & 1, w));
      if (!ok) break;
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        const int c = 2 * rd + cb;
        const uint32_t box = sm.stage() + static_cast<uint32_t>(cb * kBoxBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4_b32(box + static_cast<uint32_t>(r * 128 + ((k ^ (r & 7)) << 4)), a[32 * c + 4 * k],
                           a[32 * c + 4 * k + 1], a[32 * c + 4 * k + 2], a[32 * c + 4 * k + 3]);
      }
      fence_async_smem();
      mbar_arrive(sm.staged());
      if (leader) {  // rows past the head's last query fall outside the tensor map and are skipped
        ok = bwd_wait(sm.staged(), nround & 1, w);
        if (ok) {
          tma_reduce_add_3d(tmDQ, sm.stage(), 64 * rd, q0, wk.bh);
          tma_reduce_add_3d(tmDQ, sm.stage() + kBoxBytes, 64 * rd + 32, q0, wk.bh);
          bulk_commit();
          issued = true;
          bulk_wait_read_all();  // the staging buffer has been read
          mbar_arrive(sm.stage_free());
        }
      }
      ++nround;
    }
    if (!__all_sync(0xffffffffu, ok)) break;
  }
  if (leader && issued) bulk_wait_all();  // the reductions are complete before the CTA exits
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_sm103a(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  if ((base & 1023u) != 0u) {  // the layout has no slack for realignment: report, run nothing
    grid_dependency_wait();     // still complete only after the kernel before, like every launch here
    if (threadIdx.x == 0) atomicOr(&g_attn_status, 2u);
    return;
  }
  uint8_t* smem = smem_raw;
  const BwdSmem<D> sm{base};
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);

  if (threadIdx.x == 0) {
    mbar_init(sm.kv_full(), 1);
    for (int s = 0; s < C::kQSlots; ++s) {
      mbar_init(sm.q_full(s), 1);
      mbar_init(sm.q_empty(s), 1);
    }
    mbar_init(sm.do_full(), 1);
    mbar_init(sm.do_empty(), 1);
    mbar_init(sm.s_full(), 1);
    mbar_init(sm.dp_full(), 1);
    mbar_init(sm.p_ready(), kBM * C::kRowWGs);
    mbar_init(sm.ds_ready(), kBM * C::kRowWGs);
    mbar_init(sm.dq_full(), 1);
    mbar_init(sm.dq_free(), kBM * C::kRowWGs);
    mbar_init(sm.dsm_free(), 1);
    mbar_init(sm.done(), 1);
    mbar_init(sm.drain(), 1);
    mbar_init(sm.stat(0), kBM);
    mbar_init(sm.stat(1), kBM);
    mbar_init(sm.staged(), kBM);
    mbar_init(sm.stage_free(), 1);
    for (int h = 0; h < 2; ++h) mbar_init(sm.stat_h(1, h), kBM);
    mbar_init(sm.staged_h(1), kBM);
    mbar_init(sm.stage_free_h(1), 1);
    misc[1] = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(base + C::kMiscOff, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtx w{p.timeout_ns, misc + 1};
  // On-chip set-up is done; global memory (the statistics and the zeroed dQ
  // accumulator of the kernel before, kv_valid_len) is read from here on.
  grid_dependency_wait();
  const BwdWork wk = bwd_work(p);

  if (warp == 0) {
    if (lane == 0 && wk.n > 0) bwd_load_role<D>(sm, &tmQ, &tmK, &tmV, &tmDO, wk, w);
  } else if (warp == 1) {
    if (wk.n > 0) bwd_mma_role<D>(sm, tmem, wk, w);
  } else if (warp >= 4) {
    if constexpr (C::kRowWGs == 2) {
      bwd_row_role2<D>(sm, smem, &tmDQ, tmem, p, wk, w, (warp - 4) >> 2);
    } else if (warp < 8) {
      bwd_row_role<D>(sm, smem, tmem, p, wk, w);
    } else {
      bwd_dq_role<D>(sm, &tmDQ, tmem, p, wk, w);
    }
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

// Delta_i = sum_d dO_id O_id and lse2_i = LSE_i log2(e) per query row, padded
// to S_pad rows (+inf / 0 on padding and for rows without keys, so P = 0
// there); zeroes the fp32 dQ accumulator.  One warp per row.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep(const uint16_t* __restrict__ o, const uint16_t* __restrict__ d_o,
                                                     const float* __restrict__ lse, float* __restrict__ lse2,
                                                     float* __restrict__ delta, float* __restrict__ dq_acc, int S_q,
                                                     int S_pad, int64_t BH) {
  constexpr int kPer = D / 32;
  grid_dependency_wait();  // O and LSE come from the forward pass
  grid_launch_dependents();
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int64_t first = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t step = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = first; row < BH * S_pad; row += step) {
    const int64_t bh = row / S_pad;
    const int q = static_cast<int>(row % S_pad);
    float acc = 0.f, l2 = INFINITY;
    if (q < S_q) {
      // each lane: kPer consecutive bf16 of O and dO in one 4- or 8-byte load,
      // and the same kPer fp32 of the accumulator zeroed in one store
      const int64_t e0 = (bh * S_q + q) * D + lane * kPer;
      uint32_t ow[kPer / 2], gw[kPer / 2];
      if constexpr (kPer == 4) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(o + e0));
        const uint2 g = __ldg(reinterpret_cast<const uint2*>(d_o + e0));
        ow[0] = a.x; ow[kPer / 2 - 1] = a.y;
        gw[0] = g.x; gw[kPer / 2 - 1] = g.y;
        *reinterpret_cast<float4*>(dq_acc + e0) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        ow[0] = __ldg(reinterpret_cast<const uint32_t*>(o + e0));
        gw[0] = __ldg(reinterpret_cast<const uint32_t*>(d_o + e0));
        *reinterpret_cast<float2*>(dq_acc + e0) = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int e = 0; e < kPer / 2; ++e) {
        acc = fmaf(__uint_as_float(ow[e] << 16), __uint_as_float(gw[e] << 16), acc);
        acc = fmaf(__uint_as_float(ow[e] & 0xFFFF0000u), __uint_as_float(gw[e] & 0xFFFF0000u), acc);
      }
      const float l = __ldg(lse + bh * S_q + q);
      l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      lse2[row] = l2;
      delta[row] = q < S_q ? acc : 0.f;
    }
  }
}

// dQ = bf16(scale * accumulator), four elements per thread step.
__global__ void __launch_bounds__(256) attn_bwd_dq_convert(const float* __restrict__ dq_acc, uint16_t* __restrict__ dq,
                                                           int64_t n4, float scale) {
  grid_dependency_wait();  // the accumulator is complete once the gradient kernel is
  grid_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(dq_acc) + i);
    uint2 out;
    out.x = pack_bf16x2(a.x * scale, a.y * scale);
    out.y = pack_bf16x2(a.z * scale, a.w * scale);
    reinterpret_cast<uint2*>(dq)[i] = out;
  }
}

