// kb_backward.cu -- gradient of the causal GQA attention of a whole sequence
// (KernelBraid README, "Motivation": the policy-update step of RL training
// differentiates the same attention the rollouts ran forward).
//
// With P the row softmax of s = q.k / sqrt(128) over keys 0..i, recomputed
// from the forward's log-sum-exp, and dO the gradient of the output:
//   delta_i = dO_i . O_i                     (= sum_j P_ij dP_ij)
//   dP_ij   = dO_i . v_j
//   dS_ij   = P_ij (dP_ij - delta_i)
//   dq_i    = sum_j dS_ij k_j / sqrt(128)
//   dk_j    = sum over the group's heads and rows i >= j of dS_ij q_i / sqrt(128)
//   dv_j    = sum over the group's heads and rows i >= j of P_ij dO_i
//
// Three kernels, no atomics (every gradient element is summed by one CTA in
// one fixed order, so repeated runs give the same bits):
//   kb_bwd_delta_kernel  one warp per row: delta = rowsum(dO * O)
//   kb_bwd_dq_kernel     one CTA per (b, head, query tile): walks key tiles
//                        0..t; S = Q K^T and dP = dO V^T on the tensor core,
//                        dS in TMEM, dQ += dS K
//   kb_bwd_dkdv_kernel   one CTA per (b, kv head, key tile): walks the four
//                        heads of the group and query tiles t..n-1;
//                        S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q
// Every product uses the two forms of the forward: both operands K-major in
// shared memory (issue_qk), or A from TMEM and B MN-major (issue_pv).
#include <type_traits>

#include "kb_contract.cuh"
#include "kb_launch.h"

namespace kb {

namespace {

constexpr float kLog2e = 1.4426950408889634f;          // log2(e), to turn a natural-log lse into base 2
constexpr float kInvSqrtD = 0.088388347648318440f;     // 1 / sqrt(128)

__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 50000000ull) break;
}

// P = 2^(s c - lse2) and dS = P (dP - delta) of two adjacent columns, as
// packed f32x2 operations (the same IEEE operations, so the same bits, as the
// scalar fma, subtraction and product): `nl` and `nd` hold -lse2 and -delta.
// A masked P is zero before dS is formed, so its dS is a signed zero as in the
// scalar form.  Both values go out as one bf16 pair each.
template <bool kMask>
__device__ __forceinline__ void p_ds_pair(uint32_t s0, uint32_t s1, uint32_t dp0, uint32_t dp1, float2 c2,
                                          float2 nl, float2 nd, bool m0, bool m1, uint32_t& p_bf,
                                          uint32_t& ds_bf) {
  const float2 a = __ffma2_rn(make_float2(__uint_as_float(s0), __uint_as_float(s1)), c2, nl);
  float2 pp = make_float2(ex2_approx(a.x), ex2_approx(a.y));
  if (kMask) {
    if (m0) pp.x = 0.0f;
    if (m1) pp.y = 0.0f;
  }
  const float2 d = __fmul2_rn(pp, __fadd2_rn(make_float2(__uint_as_float(dp0), __uint_as_float(dp1)), nd));
  p_bf = pack_bf16x2(pp.x, pp.y);
  ds_bf = pack_bf16x2(d.x, d.y);
}

// Two independent products of the same shape, their K steps interleaved
// (each accumulator still takes its eight steps in ascending order): the
// tensor pipe overlaps the two dependency chains.
__device__ __forceinline__ void issue_qk_pair(uint32_t d1, uint32_t a1, uint32_t b1, uint32_t d2, uint32_t a2,
                                              uint32_t b2) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    mma_ss(d1, desc_kmajor(a1, kk, 1024u, kSlabBytes), desc_kmajor(b1, kk, 1024u, kSlabBytes), kIdescQK,
           kk > 0 ? 1u : 0u);
    mma_ss(d2, desc_kmajor(a2, kk, 1024u, kSlabBytes), desc_kmajor(b2, kk, 1024u, kSlabBytes), kIdescQK,
           kk > 0 ? 1u : 0u);
  }
}

template <int kFrom, int kTo>
__device__ __forceinline__ void issue_pv_pair(uint32_t d1, uint32_t a1_tmem, uint32_t b1, uint32_t d2,
                                              uint32_t a2_tmem, uint32_t b2, bool first) {
#pragma unroll
  for (int kk = kFrom; kk < kTo; ++kk) {
    const uint32_t acc = (first && kk == 0) ? 0u : 1u;
    mma_ts(d1, a1_tmem + static_cast<uint32_t>(kk) * 8u, desc_v(b1, kk), kIdescPV, acc);
    mma_ts(d2, a2_tmem + static_cast<uint32_t>(kk) * 8u, desc_v(b2, kk), kIdescPV, acc);
  }
}

// 16x256b loads of 32 columns (four repetitions) from two addresses, one
// wait: thread t gets lanes t/4 and t/4 + 8, columns 8r + 2(t%4) and
// 8r + 2(t%4) + 1 of repetition r in registers 4r, 4r+1 (first lane) and
// 4r+2, 4r+3 (second lane).
__device__ __forceinline__ void tmem_ld_16x256b_x4_pair_wait(uint32_t ta, uint32_t tb, uint32_t (&ra)[16],
                                                             uint32_t (&rb)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7]),
        "=r"(ra[8]), "=r"(ra[9]), "=r"(ra[10]), "=r"(ra[11]), "=r"(ra[12]), "=r"(ra[13]), "=r"(ra[14]), "=r"(ra[15]),
        "=r"(rb[0]), "=r"(rb[1]), "=r"(rb[2]), "=r"(rb[3]), "=r"(rb[4]), "=r"(rb[5]), "=r"(rb[6]), "=r"(rb[7]),
        "=r"(rb[8]), "=r"(rb[9]), "=r"(rb[10]), "=r"(rb[11]), "=r"(rb[12]), "=r"(rb[13]), "=r"(rb[14]), "=r"(rb[15])
      : "r"(ta), "r"(tb)
      : "memory");
}
// 16x128b store of 16 columns (four repetitions): thread t writes lanes t/4
// and t/4 + 8, column 4r + t%4 of repetition r, from registers 2r and 2r+1.
__device__ __forceinline__ void tmem_st_16x128b_x4(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace

// ------------------------------------------------------------------ delta

// One warp per row of 128: lane l takes elements 4l..4l+3; the four products
// are summed in pairs, then across lanes by a fixed butterfly.
__global__ void __launch_bounds__(256) kb_bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                           const __nv_bfloat16* __restrict__ dout,
                                                           float* __restrict__ delta, long long rows) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const uint2 a = reinterpret_cast<const uint2*>(o + row * kHeadDim)[lane];
  const uint2 g = reinterpret_cast<const uint2*>(dout + row * kHeadDim)[lane];
  const float p01 = __fmaf_rn(bf16_lo(a.x), bf16_lo(g.x), __fmul_rn(bf16_hi(a.x), bf16_hi(g.x)));
  const float p23 = __fmaf_rn(bf16_lo(a.y), bf16_lo(g.y), __fmul_rn(bf16_hi(a.y), bf16_hi(g.y)));
  float s = __fadd_rn(p01, p23);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, m));
  if (lane == 0) delta[row] = s;
}

// -------------------------------------------------------------- dq kernel

struct BwdQCfg {
  static constexpr int kThreads = 384;        // 8 elementwise warps, two producers, two MMA issuers
  static constexpr int kLoadWarp = 8;         // Q, dO and the K ring
  static constexpr int kMmaWarp = 9;          // TMEM allocator + S, dP issuer
  static constexpr int kDqWarp = 10;          // dQ issuer
  static constexpr int kLoadWarpV = 11;       // the V ring
  // K(j) is read by S(j) and by dQ(j), V(j) only by dP(j): the K ring frees
  // a slot after dQ(j), the V ring after S(j), dP(j), so V needs fewer slots
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kDOOff = kTileBytes;
  static constexpr uint32_t kKOff = 2 * kTileBytes;
  static constexpr uint32_t kVOff = kKOff + kKStages * kTileBytes;
  static constexpr uint32_t kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kBarQD = 0;                         // Q and dO landed
  static constexpr int kBarKFull = 1;                      // 3: K(j) landed in slot j%3
  static constexpr int kBarKEmpty = kBarKFull + kKStages;  // 3: dQ(j) done, K slot j%3 free
  static constexpr int kBarVFull = kBarKEmpty + kKStages;  // 2: V(j) landed in slot j%2
  static constexpr int kBarVEmpty = kBarVFull + kVStages;  // 2: S(j), dP(j) done, V slot j%2 free
  static constexpr int kBarSFull = kBarVEmpty + kVStages;  // S(j), dP(j) in TMEM
  static constexpr int kBarSFree = kBarSFull + 1;          // S(j) read (256 arrivals)
  static constexpr int kBarDSFull = kBarSFree + 1;         // dS(j) in TMEM (256 arrivals)
  static constexpr int kBarDQDone = kBarDSFull + 1;        // dQ += dS(j) K(j) finished
  static constexpr int kBarDrain = kBarDQDone + 1;          // 2: one per issuer
  static constexpr int kBarDPFree = kBarDrain + 2;         // dP(j) read (256 arrivals)
  static constexpr int kBarSDone = kBarDPFree + 1;         // S(j) in TMEM (kBarSFull: dP(j) too)
  static constexpr int kNumBars = kBarSDone + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
};

__global__ void __launch_bounds__(BwdQCfg::kThreads, 1)
kb_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                 const BwdArgs args) {
  using Cfg = BwdQCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) { return smem_addr(bars + i); };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // (b, h, query tile t), longest first; beyond a few waves group-major in
  // windows of two groups (the longest tiles of both groups first)
  int b, g, h, tile_rank;
  if (args.group_major) {
    constexpr int kWin = 2;
    const int BG = args.B * args.Hkv, per = args.n_tiles * kGroup, full = BG / kWin;
    const int bid = static_cast<int>(blockIdx.x);
    int w, r, wg;
    if (bid < full * kWin * per) { w = bid / (kWin * per); r = bid % (kWin * per); wg = kWin; }
    else { w = full; r = bid - full * kWin * per; wg = BG - full * kWin; }
    tile_rank = r / (wg * kGroup);
    const int rem = r % (wg * kGroup);
    const int bg = w * kWin + rem / kGroup;
    b = bg / args.Hkv;
    g = bg % args.Hkv;
    h = g * kGroup + rem % kGroup;
  } else {
    tile_rank = blockIdx.x / (args.B * args.Hq);
    const int rem = blockIdx.x % (args.B * args.Hq);
    b = rem / args.Hq;
    h = rem % args.Hq;
    g = h / kGroup;
  }
  const int t = args.n_tiles - 1 - tile_rank;
  const int n_kv = t + 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i)
      mbar_init(bar(i), (i == Cfg::kBarSFree || i == Cfg::kBarDSFull || i == Cfg::kBarDPFree) ? 256u : 1u);
    misc[1] = (*reinterpret_cast<volatile uint32_t*>(args.err) != 0) ? 1u : 0u;
    fence_mbar_init();
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(sbase + Cfg::kMiscOff, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const bool skip = (*abort_flag != 0);

  if (warp == Cfg::kLoadWarp || warp == Cfg::kLoadWarpV) {
    // ----------------------------------------------------------- producers
    // One warp per ring: Q, dO and K; V.
    const bool is_v = (warp == Cfg::kLoadWarpV);
    if (!skip) {
      const uint64_t keep = l2_policy_evict_last();
      const int stages = is_v ? Cfg::kVStages : Cfg::kKStages;
      const int full0 = is_v ? Cfg::kBarVFull : Cfg::kBarKFull;
      const int empty0 = is_v ? Cfg::kBarVEmpty : Cfg::kBarKEmpty;
      const uint32_t ring = sbase + (is_v ? Cfg::kVOff : Cfg::kKOff);
      const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
      if (lane == 0) {
        tma_prefetch_desc(tmap);
        if (!is_v) {
          tma_prefetch_desc(&tmap_q);
          tma_prefetch_desc(&tmap_do);
          mbar_arrive_expect_tx(bar(Cfg::kBarQD), 2 * kTileBytes);
          tma_load_tile(sbase + Cfg::kQOff, &tmap_q, t * kTileRows, b * args.Hq + h, bar(Cfg::kBarQD));
          tma_load_tile(sbase + Cfg::kDOOff, &tmap_do, t * kTileRows, b * args.Hq + h, bar(Cfg::kBarQD));
        }
      }
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int slot = j % stages;
        if (j >= stages)
          ok = mbar_wait(bar(empty0 + slot), ((j / stages) - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(full0 + slot), kTileBytes);
          tma_load_tile_hint(ring + slot * kTileBytes, tmap, j * kTileRows, b * args.Hkv + g, bar(full0 + slot), keep);
        }
        issued = j + 1;
      }
      if (!ok && lane == 0) {
        if (!is_v) drain_wait_b(bar(Cfg::kBarQD), 0);
        for (int x = (issued > stages ? issued - stages : 0); x < issued; ++x)
          drain_wait_b(bar(full0 + x % stages), (x / stages) & 1);
      }
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ------------------------------------------------------ S, dP issuer
    // S(j+1), dP(j+1) go out as soon as the elementwise warps have read S(j),
    // dP(j); a second thread issues the dQ products, so neither stream's
    // barrier waits leave the tensor pipe idle.
    if (lane == 0 && !skip) {
      const uint32_t q_s = sbase + Cfg::kQOff, do_s = sbase + Cfg::kDOOff;
      bool ok = mbar_wait(bar(Cfg::kBarQD), 0, abort_flag, args.err, kDevTimeoutTma);
      for (int j = 0; j < n_kv && ok; ++j) {
        const int ks = j % Cfg::kKStages, vs = j % Cfg::kVStages;
        ok = mbar_wait_hint(bar(Cfg::kBarKFull + ks), (j / Cfg::kKStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        if (ok) ok = mbar_wait_hint(bar(Cfg::kBarVFull + vs), (j / Cfg::kVStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        if (ok && j > 0) ok = mbar_wait_hint(bar(Cfg::kBarSFree), (j - 1) & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        // S's first K step goes out once S(j-1) has been read, the rest, with
        // dP's steps interleaved, once dP(j-1) has been read too
        const uint32_t k_s = sbase + Cfg::kKOff + ks * kTileBytes, v_s = sbase + Cfg::kVOff + vs * kTileBytes;
        mma_ss(tmem_base + Cfg::kColS, desc_kmajor(q_s, 0, 1024u, kSlabBytes), desc_kmajor(k_s, 0, 1024u, kSlabBytes),
               kIdescQK, 0u);
        if (j > 0) ok = mbar_wait_hint(bar(Cfg::kBarDPFree), (j - 1) & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_ss(tmem_base + Cfg::kColDP, desc_kmajor(do_s, kk, 1024u, kSlabBytes), desc_kmajor(v_s, kk, 1024u, kSlabBytes),
                 kIdescQK, kk > 0 ? 1u : 0u);
          if (kk < 7)
            mma_ss(tmem_base + Cfg::kColS, desc_kmajor(q_s, kk + 1, 1024u, kSlabBytes),
                   desc_kmajor(k_s, kk + 1, 1024u, kSlabBytes), kIdescQK, 1u);
          if (kk == 6) tc_commit(bar(Cfg::kBarSDone));             // S is complete before dP's last step
        }
        tc_commit(bar(Cfg::kBarSFull));
        tc_commit(bar(Cfg::kBarVEmpty + vs));
      }
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain));
        drain_wait_b(bar(Cfg::kBarDrain), 0);
      }
    }
  } else if (warp == Cfg::kDqWarp) {
    // ---------------------------------------------------------- dQ issuer
    // dQ(j) reads dS(j) and K(j); the K slot is released after it (S(j)
    // finished before dS(j) existed).
    if (lane == 0 && !skip) {
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        ok = mbar_wait_hint(bar(Cfg::kBarDSFull), j & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        const int ks = j % Cfg::kKStages;
        issue_pv(tmem_base + Cfg::kColDQ, tmem_base + Cfg::kColDS, sbase + Cfg::kKOff + ks * kTileBytes, j == 0);
        tc_commit(bar(Cfg::kBarDQDone));
        tc_commit(bar(Cfg::kBarKEmpty + ks));
      }
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain + 1));
        drain_wait_b(bar(Cfg::kBarDrain + 1), 0);
      }
    }
  } else {
    // ------------------------------------------------------- elementwise
    // Warp w owns TMEM lanes 32(w%4) + 16(w/4) .. +15; a thread holds rows
    // lane/4 and lane/4 + 8 of that block and, of each group of 8 keys, keys
    // 2u and 2u+1 (u = lane % 4), as the 16x256b load lays them out.
    const int lane_base = 32 * (warp & 3) + 16 * (warp >> 2);
    const uint32_t lane_off = static_cast<uint32_t>(lane_base) << 16;
    const int u = lane & 3;
    const int rA = lane_base + (lane >> 2);
    const int rB = rA + 8;
    const int iA = t * kTileRows + rA, iB = t * kTileRows + rB;       // query positions
    const bool vA = iA < args.S, vB = iB < args.S;
    const size_t row0 = (static_cast<size_t>(b) * args.Hq + h) * static_cast<size_t>(args.S);
    // rows past the sequence have zero q and dO: lse2 = 0 and delta = 0 make
    // their dS zero
    const float lseA = vA ? __fmul_rn(args.lse[row0 + iA], kLog2e) : 0.0f;
    const float lseB = vB ? __fmul_rn(args.lse[row0 + iB], kLog2e) : 0.0f;
    const float dlA = vA ? args.delta[row0 + iA] : 0.0f;
    const float dlB = vB ? args.delta[row0 + iB] : 0.0f;
    const float2 c2 = make_float2(score_scale_log2(), score_scale_log2());
    const float2 nlA = make_float2(-lseA, -lseA), nlB = make_float2(-lseB, -lseB);
    const float2 ndA = make_float2(-dlA, -dlA), ndB = make_float2(-dlB, -dlB);
    // the diagonal tile masks keys past the row; the others take no select
    auto tile_ds = [&](auto diag_tag, const uint32_t (&sv)[32], const uint32_t (&pv)[32], int half,
                       uint32_t (&ds)[32]) {
      constexpr bool kDiag = decltype(diag_tag)::value;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int key = 64 * half + 8 * r + 2 * u;                   // keys key, key + 1 within the tile
        uint32_t unused;
        p_ds_pair<kDiag>(sv[4 * r], sv[4 * r + 1], pv[4 * r], pv[4 * r + 1], c2, nlA, ndA, key > rA, key + 1 > rA,
                         unused, ds[2 * (8 * half + r)]);
        p_ds_pair<kDiag>(sv[4 * r + 2], sv[4 * r + 3], pv[4 * r + 2], pv[4 * r + 3], c2, nlB, ndB, key > rB,
                         key + 1 > rB, unused, ds[2 * (8 * half + r) + 1]);
      }
    };
    bool ok = !skip;
    for (int j = 0; j < n_kv && ok; ++j) {
      ok = mbar_wait_hint(bar(Cfg::kBarSDone), j & 1, abort_flag, args.err, kDevTimeoutMma);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool diag = (j == n_kv - 1);
      uint32_t ds[32];
      // all of S(j) and dP(j) into registers first, so S(j+1), dP(j+1) can be
      // issued while this tile's dS is computed: S as soon as it is complete
      // (before dP's last step), released on its own barrier so S(j+1) can
      // start while dP is still being read
      uint32_t sv0[32], pv0[32], sv1[32], pv1[32];
      tmem_ld_16x256b_x8_pair_wait(tmem_base + Cfg::kColS + lane_off, tmem_base + Cfg::kColS + lane_off + 64u, sv0,
                                   sv1);
      tc_fence_before();
      mbar_arrive(bar(Cfg::kBarSFree));                              // S(j) fully read
      ok = mbar_wait_hint(bar(Cfg::kBarSFull), j & 1, abort_flag, args.err, kDevTimeoutMma);   // dP(j) too
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      tmem_ld_16x256b_x8_pair_wait(tmem_base + Cfg::kColDP + lane_off, tmem_base + Cfg::kColDP + lane_off + 64u, pv0,
                                   pv1);
      tc_fence_before();
      mbar_arrive(bar(Cfg::kBarDPFree));                             // dP(j) fully read
      if (diag) {
        tile_ds(std::true_type{}, sv0, pv0, 0, ds);
        tile_ds(std::true_type{}, sv1, pv1, 1, ds);
      } else {
        tile_ds(std::false_type{}, sv0, pv0, 0, ds);
        tile_ds(std::false_type{}, sv1, pv1, 1, ds);
      }
      if (j > 0) {                                                   // dQ(j-1) has read dS(j-1)
        ok = mbar_wait(bar(Cfg::kBarDQDone), (j - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st_16x128b_x16(tmem_base + Cfg::kColDS + lane_off, ds);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Cfg::kBarDSFull));
    }
    if (ok) ok = mbar_wait(bar(Cfg::kBarDQDone), (n_kv - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* base = static_cast<__nv_bfloat16*>(args.dq) + row0 * kHeadDim;
      uint32_t* dA = reinterpret_cast<uint32_t*>(base + static_cast<size_t>(vA ? iA : 0) * kHeadDim);
      uint32_t* dB = reinterpret_cast<uint32_t*>(base + static_cast<size_t>(vB ? iB : 0) * kHeadDim);
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
        tmem_ld_16x256b_x8_wait(tmem_base + Cfg::kColDQ + lane_off + 64u * half, v);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int col = 64 * half + 8 * r + 2 * u;
          const uint32_t wa = pack_bf16x2(__fmul_rn(__uint_as_float(v[4 * r]), kInvSqrtD),
                                          __fmul_rn(__uint_as_float(v[4 * r + 1]), kInvSqrtD));
          const uint32_t wb = pack_bf16x2(__fmul_rn(__uint_as_float(v[4 * r + 2]), kInvSqrtD),
                                          __fmul_rn(__uint_as_float(v[4 * r + 3]), kInvSqrtD));
          if (vA) dA[col >> 1] = wa;
          if (vB) dB[col >> 1] = wb;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ----------------------------------------------------------- dk/dv kernel

struct BwdKVCfg {
  static constexpr int kThreads = 320;
  static constexpr int kLoadWarp = 8;
  static constexpr int kMmaWarp = 9;
  static constexpr int kStages = 2;           // Q/dO ring
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColST = 0, kColDPT = 128, kColDV = 256, kColDK = 384;
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kTileBytes;
  static constexpr uint32_t kQOff = 2 * kTileBytes;                   // slot s: Q at kQOff + s*2*tile,
  static constexpr uint32_t kSlotBytes = 2 * kTileBytes;              //         dO right after it
  static constexpr uint32_t kVecOff = kQOff + kStages * kSlotBytes;   // slot s: -lse2[128], -delta[128]
  static constexpr uint32_t kVecBytes = 2 * 128 * 4;
  static constexpr uint32_t kBarOff = kVecOff + kStages * kVecBytes;
  static constexpr int kBarKV = 0;                                    // K(jt), V(jt) landed
  static constexpr int kBarQDFull = 1;                                // 2: Q, dO of step s landed
  static constexpr int kBarQDEmpty = kBarQDFull + kStages;            // 2: dV, dK of step s done
  static constexpr int kBarVecFull = kBarQDEmpty + kStages;           // 2: lse2, delta of step s (32 arrivals)
  static constexpr int kBarSTFull = kBarVecFull + kStages;            // S^T, dP^T of step s in TMEM
  static constexpr int kBarPDSFull = kBarSTFull + 1;                  // 4: P^T, dS^T of query quarter 0..3
                                                                      //    stored (256 arrivals each)
  static constexpr int kBarDone = kBarPDSFull + 4;                    // every dV, dK product finished
  static constexpr int kBarDrain = kBarDone + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
};

__global__ void __launch_bounds__(BwdKVCfg::kThreads, 1)
kb_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                   const BwdArgs args) {
  using Cfg = BwdKVCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) { return smem_addr(bars + i); };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // (b, kv head g, key tile jt) in windows of two groups, (b, g) windows
  // slowest so resident CTAs share the groups' q and dO in L2; within a
  // window the longest key tiles (jt = 0) of both groups first, so the last
  // window's longest CTAs start early and the launch ends on short ones
  int bg, jt;
  {
    constexpr int kWin = 2;
    const int BG = args.B * args.Hkv, n = args.n_tiles, full = BG / kWin;
    const int bid = static_cast<int>(blockIdx.x);
    int w, r, wg;
    if (bid < full * kWin * n) { w = bid / (kWin * n); r = bid % (kWin * n); wg = kWin; }
    else { w = full; r = bid - full * kWin * n; wg = BG - full * kWin; }
    jt = r / wg;
    bg = w * kWin + r % wg;
  }
  const int b = bg / args.Hkv;
  const int g = bg % args.Hkv;
  const int n_q = args.n_tiles - jt;                  // query tiles jt..n-1 see this key tile
  const int n_steps = kGroup * n_q;                   // step s: head g*4 + s / n_q, query tile jt + s % n_q

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i) {
      uint32_t count = 1u;
      if (i >= Cfg::kBarPDSFull && i < Cfg::kBarPDSFull + 4) count = 256u;
      if (i >= Cfg::kBarVecFull && i < Cfg::kBarVecFull + Cfg::kStages) count = 32u;
      mbar_init(bar(i), count);
    }
    misc[1] = (*reinterpret_cast<volatile uint32_t*>(args.err) != 0) ? 1u : 0u;
    fence_mbar_init();
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(sbase + Cfg::kMiscOff, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const bool skip = (*abort_flag != 0);

  if (warp == Cfg::kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (!skip) {
      const uint64_t keep = l2_policy_evict_last();
      if (lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_do);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        mbar_arrive_expect_tx(bar(Cfg::kBarKV), 2 * kTileBytes);
        tma_load_tile(sbase + Cfg::kKOff, &tmap_k, jt * kTileRows, b * args.Hkv + g, bar(Cfg::kBarKV));
        tma_load_tile(sbase + Cfg::kVOff, &tmap_v, jt * kTileRows, b * args.Hkv + g, bar(Cfg::kBarKV));
      }
      int issued = 0;
      bool ok = true;
      for (int s = 0; s < n_steps; ++s) {
        const int slot = s % Cfg::kStages;
        const int h = g * kGroup + s / n_q;
        const int it = jt + s % n_q;
        if (s >= Cfg::kStages)
          ok = mbar_wait(bar(Cfg::kBarQDEmpty + slot), ((s / Cfg::kStages) - 1) & 1, abort_flag, args.err,
                         kDevTimeoutSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t dst = sbase + Cfg::kQOff + slot * Cfg::kSlotBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(Cfg::kBarQDFull + slot), 2 * kTileBytes);
          tma_load_tile_hint(dst, &tmap_q, it * kTileRows, b * args.Hq + h, bar(Cfg::kBarQDFull + slot), keep);
          tma_load_tile_hint(dst + kTileBytes, &tmap_do, it * kTileRows, b * args.Hq + h,
                             bar(Cfg::kBarQDFull + slot), keep);
        }
        issued = s + 1;
        // -lse (base 2) and -delta of the step's 128 query rows; rows past the
        // sequence get -lse2 = -inf, so their P (and dS) is exactly zero
        float* vec = reinterpret_cast<float*>(smem + Cfg::kVecOff + slot * Cfg::kVecBytes);
        const size_t row0 = (static_cast<size_t>(b) * args.Hq + h) * static_cast<size_t>(args.S);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = 4 * lane + e;
          const int i = it * kTileRows + q;
          const bool valid = i < args.S;
          vec[q] = valid ? -__fmul_rn(args.lse[row0 + i], kLog2e) : __int_as_float(0xFF800000);
          vec[128 + q] = valid ? -args.delta[row0 + i] : -0.0f;
        }
        mbar_arrive(bar(Cfg::kBarVecFull + slot));
      }
      if (!ok && lane == 0) {
        drain_wait_b(bar(Cfg::kBarKV), 0);
        for (int x = (issued > Cfg::kStages ? issued - Cfg::kStages : 0); x < issued; ++x)
          drain_wait_b(bar(Cfg::kBarQDFull + x % Cfg::kStages), (x / Cfg::kStages) & 1);
      }
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // per step: S^T = K Q^T, dP^T = V dO^T, then for each quarter of the
    // query columns (32 queries), once its P^T and dS^T are stored, K steps
    // 2q and 2q+1 of dV += P^T dO and dK += dS^T Q.  A quarter's steps read
    // only the columns that quarter wrote, so they run while the next quarter
    // is computed.  P^T and dS^T overwrite S^T and dP^T, whose next values are
    // issued after these products (in issue order).
    if (lane == 0 && !skip) {
      bool ok = mbar_wait(bar(Cfg::kBarKV), 0, abort_flag, args.err, kDevTimeoutTma);
      for (int s = 0; s < n_steps && ok; ++s) {
        const int slot = s % Cfg::kStages;
        const uint32_t q_s = sbase + Cfg::kQOff + slot * Cfg::kSlotBytes;
        const uint32_t do_s = q_s + kTileBytes;
        ok = mbar_wait_hint(bar(Cfg::kBarQDFull + slot), (s / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        if (!ok) break;
        tc_fence_after();
        issue_qk_pair(tmem_base + Cfg::kColST, sbase + Cfg::kKOff, q_s, tmem_base + Cfg::kColDPT, sbase + Cfg::kVOff,
                      do_s);
        tc_commit(bar(Cfg::kBarSTFull));
        ok = mbar_wait_hint(bar(Cfg::kBarPDSFull), s & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        issue_pv_pair<0, 2>(tmem_base + Cfg::kColDV, tmem_base + Cfg::kColST, do_s, tmem_base + Cfg::kColDK,
                            tmem_base + Cfg::kColDPT, q_s, s == 0);
        ok = mbar_wait_hint(bar(Cfg::kBarPDSFull + 1), s & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        issue_pv_pair<2, 4>(tmem_base + Cfg::kColDV, tmem_base + Cfg::kColST, do_s, tmem_base + Cfg::kColDK,
                            tmem_base + Cfg::kColDPT, q_s, false);
        ok = mbar_wait_hint(bar(Cfg::kBarPDSFull + 2), s & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        issue_pv_pair<4, 6>(tmem_base + Cfg::kColDV, tmem_base + Cfg::kColST, do_s, tmem_base + Cfg::kColDK,
                            tmem_base + Cfg::kColDPT, q_s, false);
        ok = mbar_wait_hint(bar(Cfg::kBarPDSFull + 3), s & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        issue_pv_pair<6, 8>(tmem_base + Cfg::kColDV, tmem_base + Cfg::kColST, do_s, tmem_base + Cfg::kColDK,
                            tmem_base + Cfg::kColDPT, q_s, false);
        tc_commit(bar(Cfg::kBarQDEmpty + slot));
      }
      if (ok) tc_commit(bar(Cfg::kBarDone));
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain));
        drain_wait_b(bar(Cfg::kBarDrain), 0);
      }
    }
  } else {
    // ------------------------------------------------------- elementwise
    // rows are keys (lanes as in the dq kernel), columns are query rows
    const int lane_base = 32 * (warp & 3) + 16 * (warp >> 2);
    const uint32_t lane_off = static_cast<uint32_t>(lane_base) << 16;
    const int u = lane & 3;
    const int rA = lane_base + (lane >> 2);
    const int rB = rA + 8;
    const float2 c2 = make_float2(score_scale_log2(), score_scale_log2());
    // one query quarter: the diagonal step masks keys past the query, the
    // others take no select
    auto quarter = [&](auto diag_tag, const uint32_t (&sv)[16], const uint32_t (&pv)[16], const float* vnl,
                       const float* vnd, int qt, uint32_t (&pp)[8], uint32_t (&dd)[8]) {
      constexpr bool kDiag = decltype(diag_tag)::value;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int qc = 32 * qt + 8 * r + 2 * u;                      // query rows qc, qc + 1 within their tile
        const float2 nl = *reinterpret_cast<const float2*>(vnl + qc);
        const float2 nd = *reinterpret_cast<const float2*>(vnd + qc);
        p_ds_pair<kDiag>(sv[4 * r], sv[4 * r + 1], pv[4 * r], pv[4 * r + 1], c2, nl, nd, rA > qc, rA > qc + 1,
                         pp[2 * r], dd[2 * r]);
        p_ds_pair<kDiag>(sv[4 * r + 2], sv[4 * r + 3], pv[4 * r + 2], pv[4 * r + 3], c2, nl, nd, rB > qc,
                         rB > qc + 1, pp[2 * r + 1], dd[2 * r + 1]);
      }
    };
    bool ok = !skip;
    for (int s = 0; s < n_steps && ok; ++s) {
      const int slot = s % Cfg::kStages;
      const bool diag = (s % n_q) == 0;                              // query tile jt: keys past the row masked
      ok = mbar_wait_hint(bar(Cfg::kBarSTFull), s & 1, abort_flag, args.err, kDevTimeoutMma);
      if (ok) ok = mbar_wait_hint(bar(Cfg::kBarVecFull + slot), (s / Cfg::kStages) & 1, abort_flag, args.err,
                             kDevTimeoutTma);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* vnl = reinterpret_cast<const float*>(smem + Cfg::kVecOff + slot * Cfg::kVecBytes);
      const float* vnd = vnl + 128;
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {                                 // query quarter: 32 query columns
        uint32_t sv[16], pv[16];
        tmem_ld_16x256b_x4_pair_wait(tmem_base + Cfg::kColST + lane_off + 32u * qt,
                                     tmem_base + Cfg::kColDPT + lane_off + 32u * qt, sv, pv);
        uint32_t pp[8], dd[8];
        if (diag) quarter(std::true_type{}, sv, pv, vnl, vnd, qt, pp, dd);
        else quarter(std::false_type{}, sv, pv, vnl, vnd, qt, pp, dd);
        // bf16 pairs of query columns 32*qt.. go to columns 16*qt.. of the
        // same buffers; those fp32 columns were read in this quarter or an
        // earlier one
        tmem_st_16x128b_x4(tmem_base + Cfg::kColST + lane_off + 16u * qt, pp);
        tmem_st_16x128b_x4(tmem_base + Cfg::kColDPT + lane_off + 16u * qt, dd);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(Cfg::kBarPDSFull + qt));
      }
    }
    if (ok) ok = mbar_wait(bar(Cfg::kBarDone), 0, abort_flag, args.err, kDevTimeoutMma);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const int jA = jt * kTileRows + rA, jB = jt * kTileRows + rB;
      const bool vA = jA < args.S, vB = jB < args.S;
      const size_t kv0 = (static_cast<size_t>(b) * args.Hkv + g) * static_cast<size_t>(args.S);
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {                      // 0: dv, 1: dk (scaled by 1/sqrt(128))
        __nv_bfloat16* base = static_cast<__nv_bfloat16*>(which ? args.dk : args.dv) + kv0 * kHeadDim;
        uint32_t* oA = reinterpret_cast<uint32_t*>(base + static_cast<size_t>(vA ? jA : 0) * kHeadDim);
        uint32_t* oB = reinterpret_cast<uint32_t*>(base + static_cast<size_t>(vB ? jB : 0) * kHeadDim);
        const float sc = which ? kInvSqrtD : 1.0f;
        const uint32_t col0 = which ? Cfg::kColDK : Cfg::kColDV;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          tmem_ld_16x256b_x8_wait(tmem_base + col0 + lane_off + 64u * half, v);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int col = 64 * half + 8 * r + 2 * u;
            const uint32_t wa = pack_bf16x2(__fmul_rn(__uint_as_float(v[4 * r]), sc),
                                            __fmul_rn(__uint_as_float(v[4 * r + 1]), sc));
            const uint32_t wb = pack_bf16x2(__fmul_rn(__uint_as_float(v[4 * r + 2]), sc),
                                            __fmul_rn(__uint_as_float(v[4 * r + 3]), sc));
            if (vA) oA[col >> 1] = wa;
            if (vB) oB[col >> 1] = wb;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// --------------------------------------------------------------- launcher

cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t s) {
  static_assert(BwdQCfg::kSmemBytes <= 227u * 1024u, "shared memory budget (dq)");
  static_assert(BwdKVCfg::kSmemBytes <= 227u * 1024u, "shared memory budget (dk, dv)");
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kb_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(BwdQCfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kb_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(BwdKVCfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const long long rows = static_cast<long long>(a.B) * a.Hq * a.S;
  kb_bwd_delta_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.delta, rows);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long grid_q = static_cast<long long>(a.n_tiles) * a.B * a.Hq;
  kb_bwd_dq_kernel<<<static_cast<unsigned>(grid_q), BwdQCfg::kThreads, BwdQCfg::kSmemBytes, s>>>(tq, tk, tv, tdo, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long grid_kv = static_cast<long long>(a.n_tiles) * a.B * a.Hkv;
  kb_bwd_dkdv_kernel<<<static_cast<unsigned>(grid_kv), BwdKVCfg::kThreads, BwdKVCfg::kSmemBytes, s>>>(tq, tk, tv,
                                                                                                     tdo, a);
  return cudaGetLastError();
}

}  // namespace kb
