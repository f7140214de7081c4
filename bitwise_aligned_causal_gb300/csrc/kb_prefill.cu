// kb_prefill.cu -- causal GQA forward for a block of query rows against a KV
// cache: full-sequence prefill (start = 0) and partitioned/chunked forward
// (start > 0) are the same kernel (KernelBraid README, "Method": the
// numerical contract connects full-sequence prefill and partitioned forward
// execution; "Usage": causal full-sequence forward).
//
// One CTA owns NQ query tiles of 128 rows at the same absolute tile t (NQ
// heads of one GQA group) and walks KV tiles 0..t once, sharing each K/V tile
// between its query tiles.  Roles:
//   warps 0 .. 4*NQ-1  softmax: warpgroup qi owns query tile qi, thread = row
//   warp  4*NQ         TMA producer (one lane): Q once, then K_j, V_j
//   warp  4*NQ+1       TMEM allocator + MMA issuer (one lane)
// TMEM per query tile: S (128 fp32 columns; P overwrites its first 64 as
// bf16 pairs) and O (128 fp32 columns).
#include "kb_contract.cuh"
#include "kb_launch.h"

namespace kb {

template <int NQ>
struct PrefillCfg {
  static constexpr int kSoftmaxWarps = 4 * NQ;
  static constexpr int kLoadWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
  static constexpr int kStages = (NQ == 1) ? 1 : 2;
  static constexpr uint32_t kTmemCols = (NQ == 1) ? 256u : 512u;
  // Registers are split evenly over the SM's four sub-partitions, so a CTA of
  // 10 warps (3 on some sub-partition) gets at most 168 per thread, as do two
  // resident CTAs of 6 warps.
  static constexpr int kMinBlocks = (NQ == 1) ? 2 : 1;

  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = kQOff + NQ * kTileBytes;
  static constexpr uint32_t kVOff = kKOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kVOff + kStages * kTileBytes;
  // barrier indices
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 1;
  static constexpr int kBarKEmpty = kBarKFull + kStages;
  static constexpr int kBarVFull = kBarKEmpty + kStages;
  static constexpr int kBarVEmpty = kBarVFull + kStages;
  static constexpr int kBarSFull = kBarVEmpty + kStages;
  static constexpr int kBarPFull = kBarSFull + NQ;
  static constexpr int kBarOFull = kBarPFull + NQ;
  static constexpr int kBarVReady = kBarOFull + NQ;         // last V tile with its tail zeroed (paged)
  static constexpr int kBarDrain = kBarVReady + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;  // [0] tmem base, [1] abort flag
  static constexpr uint32_t kSmemUsed = kMiscOff + 16;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;      // slack for 1024-byte alignment
};

// Short bounded wait used only on the abort path, to let copies and MMAs
// already in flight land before the CTA releases its memory.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 50000000ull) break;
}

template <int NQ>
__global__ void __launch_bounds__(PrefillCfg<NQ>::kThreads, PrefillCfg<NQ>::kMinBlocks)
kb_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs args) {
  using Cfg = PrefillCfg<NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) { return smem_addr(bars + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work unit: longest query tiles first; neighbouring CTAs share (b, t) so
  // the heads of one GQA group hit the same K/V tiles in L2 together.
  const int units_per_bt = args.Hq / NQ;
  const int tile_rank = blockIdx.x / (args.B * units_per_bt);
  const int rem = blockIdx.x % (args.B * units_per_bt);
  const int b = rem / units_per_bt;
  const int h0 = (rem % units_per_bt) * NQ;
  const int g = h0 / kGroup;
  // this sequence's query rows: positions start .. start+L-1 (per sequence
  // in a ragged batch, where L is only the row stride of q and o)
  int start = args.start, L = args.L, first_tile = args.first_tile, n_tiles = args.n_tiles;
  if (args.starts != nullptr) {
    start = args.starts[b];
    L = args.lens[b];
    if (start < 0 || L < 0 || L > args.L || start + L > args.kv_cap) {
      if (threadIdx.x == 0) atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
      return;
    }
    if (L == 0) return;
    first_tile = start / kTileRows;
    n_tiles = (start + L - 1) / kTileRows - first_tile + 1;
  }
  if (tile_rank >= n_tiles) return;                                // grid sized for the longest sequence
  const int t = first_tile + n_tiles - 1 - tile_rank;              // absolute query tile
  const int n_kv = t + 1;                                          // C1: KV tiles 0..t

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i) {
      uint32_t count = 1;
      if (i >= Cfg::kBarPFull && i < Cfg::kBarPFull + NQ) count = 128;
      mbar_init(bar(i), count);
    }
    // an earlier CTA already gave up: this one only allocates and frees TMEM
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

  const bool paged = args.block_table != nullptr;
  const int kv_len = start + L;                                    // keys at or beyond kv_len are never used
  // the K/V map ends at kv_len only for a contiguous, uniform batch; else the
  // last tile's V rows past kv_len are zeroed in shared memory
  const bool zero_tail = paged || (args.starts != nullptr);
  if (warp == Cfg::kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (!skip) {
      const uint64_t keep = l2_policy_evict_last();
      if (lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        const int yq = t * kTileRows - start;           // may be negative: zero-filled rows
        mbar_arrive_expect_tx(bar(Cfg::kBarQFull), NQ * kTileBytes);
        for (int qi = 0; qi < NQ; ++qi) {
          const int zq = b * args.Hq + h0 + qi;
          const uint32_t dst = sbase + Cfg::kQOff + qi * kTileBytes;
          tma_load_tile(dst, &tmap_q, yq, zq, bar(Cfg::kBarQFull));
        }
      }
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int slot = j % Cfg::kStages;
        const uint32_t use = j / Cfg::kStages;
        // key tile j: rows of the K/V map and plane (a page of a paged pool)
        int row = j * kTileKeys, plane = b * args.Hkv + g;
        if (paged && lane == 0) {
          int pg = args.block_table[static_cast<size_t>(b) * args.pages_per_seq + row / args.page_size];
          if (pg < 0 || pg >= args.num_pages) {
            atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
            pg = args.num_pages;       // beyond the map: the TMA unit reads zeros
          }
          row = row % args.page_size;
          plane = pg * args.Hkv + g;
        }
        if (j >= Cfg::kStages)
          ok = mbar_wait(bar(Cfg::kBarKEmpty + slot), (use - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t kdst = sbase + Cfg::kKOff + slot * kTileBytes;
          mbar_arrive_expect_tx(bar(Cfg::kBarKFull + slot), kTileBytes);
          tma_load_tile_hint(kdst, &tmap_k, row, plane, bar(Cfg::kBarKFull + slot), keep);
        }
        issued = 2 * j + 1;
        if (j >= Cfg::kStages)
          ok = mbar_wait(bar(Cfg::kBarVEmpty + slot), (use - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t vdst = sbase + Cfg::kVOff + slot * kTileBytes;
          mbar_arrive_expect_tx(bar(Cfg::kBarVFull + slot), kTileBytes);
          tma_load_tile_hint(vdst, &tmap_v, row, plane, bar(Cfg::kBarVFull + slot), keep);
        }
        issued = 2 * j + 2;
      }
      if (ok && zero_tail) {
        // V rows past kv_len in the last tile may hold anything (a page's
        // unused part, another position's data, NaN): zero them so P = 0 adds
        // nothing.
        const int jl = n_kv - 1;
        const int slot = jl % Cfg::kStages;
        ok = mbar_wait(bar(Cfg::kBarVFull + slot), (jl / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          uint8_t* vt = smem + Cfg::kVOff + slot * kTileBytes;
          const int tail_from = min(kTileKeys, kv_len - jl * kTileKeys);
          for (int idx = tail_from * 16 + lane; idx < kTileKeys * 16; idx += 32) {
            const int vr = idx >> 4;
            const int c = idx & 15;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kSlabBytes + (vr >> 3) * 1024 + (vr & 7) * 128 +
                                      (((c & 7) ^ (vr & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(Cfg::kBarVReady));
        }
      }
      if (!ok && lane == 0) {
        // let every copy already issued land before shared memory is released
        drain_wait(bar(Cfg::kBarQFull), 0);
        for (int x = (issued > 2 * Cfg::kStages ? issued - 2 * Cfg::kStages : 0); x < issued; ++x) {
          const int j = x >> 1;
          const int slot = j % Cfg::kStages;
          const uint32_t use = j / Cfg::kStages;
          drain_wait(bar(((x & 1) ? Cfg::kBarVFull : Cfg::kBarKFull) + slot), use & 1);
        }
      }
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // Issue order (NQ = 2): S0(0) S1(0) | O0+=P0V(0) S0(1) O1+=P1V(0) S1(1) |
    // O0+=P0V(1) S0(2) ...  so each query tile's softmax overlaps the other
    // tile's two products.  P of a query tile lives in the first 64 columns
    // of its S buffer; the next S of that tile is issued after its P V, and
    // tcgen05.mma instructions from one thread execute in issue order.
    if (lane == 0 && !skip) {
      bool ok = mbar_wait(bar(Cfg::kBarQFull), 0, abort_flag, args.err, kDevTimeoutTma);
      if (ok) ok = mbar_wait(bar(Cfg::kBarKFull), 0, abort_flag, args.err, kDevTimeoutTma);
      if (ok) {
        tc_fence_after();
        for (int qi = 0; qi < NQ; ++qi) {
          issue_qk(tmem_base + qi * 256u, sbase + Cfg::kQOff + qi * kTileBytes, 1024u, kSlabBytes, sbase + Cfg::kKOff);
          tc_commit(bar(Cfg::kBarSFull + qi));
        }
        tc_commit(bar(Cfg::kBarKEmpty));
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int slot = j % Cfg::kStages;
        const int nslot = (j + 1) % Cfg::kStages;
        if (zero_tail && j == n_kv - 1)
          ok = mbar_wait(bar(Cfg::kBarVReady), 0, abort_flag, args.err, kDevTimeoutTma);
        else
          ok = mbar_wait(bar(Cfg::kBarVFull + slot), (j / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        for (int qi = 0; qi < NQ && ok; ++qi) {
          ok = mbar_wait(bar(Cfg::kBarPFull + qi), j & 1, abort_flag, args.err, kDevTimeoutSoftmax);
          if (!ok) break;
          tc_fence_after();
          issue_pv(tmem_base + qi * 256u + 128u, tmem_base + qi * 256u, sbase + Cfg::kVOff + slot * kTileBytes,
                   j == 0);
          tc_commit(bar(Cfg::kBarOFull + qi));
          if (qi == NQ - 1) tc_commit(bar(Cfg::kBarVEmpty + slot));
          if (j + 1 < n_kv) {
            if (qi == 0) {
              ok = mbar_wait(bar(Cfg::kBarKFull + nslot), ((j + 1) / Cfg::kStages) & 1, abort_flag, args.err,
                             kDevTimeoutTma);
              if (!ok) break;
              tc_fence_after();
            }
            issue_qk(tmem_base + qi * 256u, sbase + Cfg::kQOff + qi * kTileBytes, 1024u, kSlabBytes,
                     sbase + Cfg::kKOff + nslot * kTileBytes);
            tc_commit(bar(Cfg::kBarSFull + qi));
            if (qi == NQ - 1) tc_commit(bar(Cfg::kBarKEmpty + nslot));
          }
        }
      }
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain));   // arrives once every MMA issued so far has finished
        drain_wait(bar(Cfg::kBarDrain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int qi = warp >> 2;
    const int r = (warp & 3) * 32 + lane;           // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tmem_base + qi * 256u + lane_off;
    const uint32_t o_tmem = s_tmem + 128u;
    RowState st = row_state_init();
    bool ok = !skip;
    for (int j = 0; j < n_kv && ok; ++j) {
      ok = mbar_wait(bar(Cfg::kBarSFull + qi), j & 1, abort_flag, args.err, kDevTimeoutMma);
      ok = __all_sync(0xffffffffu, ok);   // keep the warp converged for tcgen05.ld/st
      if (!ok) break;
      tc_fence_after();
      uint32_t s[128];
      tmem_ld128_wait(s_tmem, s);
      uint32_t p[64];
      const float alpha = (j == n_kv - 1) ? row_softmax_tile<true>(s, r + 1, st, p)   // diagonal tile: causal mask
                                          : row_softmax_tile<false>(s, kTileKeys, st, p);
      if (j > 0) {
        ok = mbar_wait(bar(Cfg::kBarOFull + qi), (j - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32_wait(o_tmem + c * 32u, o);
            rescale32(o, alpha);
            tmem_st32(o_tmem + c * 32u, o);
          }
        }
      }
      {
        uint32_t p0[32], p1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) { p0[i] = p[i]; p1[i] = p[32 + i]; }
        tmem_st32(s_tmem, p0);
        tmem_st32(s_tmem + 32u, p1);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Cfg::kBarPFull + qi));
    }
    if (ok) ok = mbar_wait(bar(Cfg::kBarOFull + qi), (n_kv - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const int pos = t * kTileRows + r;
      const int i = pos - start;
      const bool store = (i >= 0) && (i < L);
      const float inv_l = row_inv_l(st);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) +
                                            ((static_cast<size_t>(b) * args.Hq + h0 + qi) * args.L + (store ? i : 0)) *
                                                kHeadDim);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32], w[16];
        tmem_ld32_wait(o_tmem + c * 32u, o);
        normalise32(o, inv_l, w);
        if (store) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[c * 4 + v4] = make_uint4(w[4 * v4 + 0], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
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

template <int NQ>
static cudaError_t launch_prefill_nq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const PrefillArgs& a, cudaStream_t s) {
  using Cfg = PrefillCfg<NQ>;
  static_assert(Cfg::kSmemUsed <= 227u * 1024u, "shared memory budget");
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kb_prefill_kernel<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const long long grid = static_cast<long long>(a.n_tiles) * a.B * (a.Hq / NQ);
  kb_prefill_kernel<NQ><<<static_cast<unsigned>(grid), Cfg::kThreads, Cfg::kSmemBytes, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

cudaError_t launch_prefill(int q_tiles_per_cta, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillArgs& a, cudaStream_t s) {
  if (q_tiles_per_cta == 1) return launch_prefill_nq<1>(tq, tk, tv, a, s);
  return launch_prefill_nq<2>(tq, tk, tv, a, s);
}

}  // namespace kb
