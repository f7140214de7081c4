// kb_decode.cu -- query rows packed by GQA group: one-token decode (KernelBraid
// README, "Usage": unified_decode over the same KV context, whose output must
// equal the prefill row bit for bit; "Features": one query token per decode
// call) and chunks of up to 32 query rows against a KV cache (README
// "Method": partitioned forward execution), on a contiguous or a paged cache.
//
// One CTA per (sub-chunk, batch, KV head).  The four query heads of the GQA
// group and the sub-chunk's rows are packed into the rows of the M=128 MMA
// (row m = head i * Lc + query row r), so the CTA issues the very same
// tcgen05.mma shape, k-order and row softmax as prefill and every packed row
// reproduces the prefill row exactly, while K and V are read once per KV head.
// A sub-chunk never crosses a 128-position tile boundary, so all its rows end
// on the same KV tile.  K/V tiles stream through a three-deep TMA ring; S has
// three TMEM buffers, so the next two Q K^T products run ahead of the softmax
// (P of a tile lives in its S buffer until that tile's P V has finished).
//   warps 0..NS-1  softmax (TMEM lanes 32w..32w+31; NS = 1 narrow, 4 wide)
//   warp  NS       TMA producer (lane 0 issues; the warp zeroes a V tail)
//   warp  NS+1     TMEM allocator + MMA issuer (one lane)
// Narrow (at most 8 packed rows): Q is one 8-row swizzle atom per d-slab and
// the row groups 8..127 of the MMA alias it (stride-byte-offset 0).
#include "kb_contract.cuh"
#include "kb_launch.h"

namespace kb {

template <bool kWide>
struct PackedCfg {
  static constexpr int kSoftmaxWarps = kWide ? 4 : 1;
  static constexpr int kProdWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
  static constexpr int kStages = 3;
  static constexpr int kQRows = kWide ? 128 : 8;
  static constexpr int kSBufs = 3;
  static constexpr uint32_t kTmemCols = 512;                  // S0, S1, S2, O (128 columns each)
  static constexpr uint32_t kOCol = kSBufs * 128u;
  static constexpr uint32_t kQSlab = kQRows * 128;            // bytes of one 64-column slab of Q
  static constexpr uint32_t kQSbo = kWide ? 1024u : 0u;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = 2 * kQSlab;
  static constexpr uint32_t kVOff = kKOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kBarKFull = 0;
  static constexpr int kBarKEmpty = kBarKFull + kStages;
  static constexpr int kBarVFull = kBarKEmpty + kStages;
  static constexpr int kBarVEmpty = kBarVFull + kStages;
  static constexpr int kBarSFull = kBarVEmpty + kStages;   // one per S buffer
  static constexpr int kBarPFull = kBarSFull + kSBufs;     // one per S buffer: P of a tile using it written
  static constexpr int kBarOFull = kBarPFull + kSBufs;     // one per S buffer: P V of a tile using it done
  static constexpr int kBarVReady = kBarOFull + kSBufs;    // last V tile with its tail zeroed
  static constexpr int kBarDrain = kBarVReady + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemUsed = kMiscOff + 16;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
};

__device__ __forceinline__ void packed_drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 50000000ull) break;
}

// Row of the K/V tensor map and plane of key tile j of sequence b, KV head g.
__device__ __forceinline__ void kv_tile_coords(const PackedArgs& a, int b, int g, int j, int& row, int& plane) {
  if (a.block_table == nullptr) {
    row = j * kTileKeys;
    plane = b * a.Hkv + g;
    return;
  }
  const int key = j * kTileKeys;
  int pg = a.block_table[static_cast<size_t>(b) * a.pages_per_seq + key / a.page_size];
  if (pg < 0 || pg >= a.num_pages) {
    atomicCAS(a.err, 0u, static_cast<uint32_t>(kDevBadInput));
    pg = a.num_pages;          // beyond the map: the TMA unit reads zeros
  }
  row = key % a.page_size;
  plane = pg * a.Hkv + g;
}

template <bool kWide>
__global__ void __launch_bounds__(PackedCfg<kWide>::kThreads, 1)
kb_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const PackedArgs args) {
  using Cfg = PackedCfg<kWide>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) { return smem_addr(bars + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = args.B * args.Hkv;
  const int seg = (args.seg_tiles > 0) ? static_cast<int>(blockIdx.x) / (args.n_sub * bh) : 0;
  const int cta = (args.seg_tiles > 0) ? static_cast<int>(blockIdx.x) % (args.n_sub * bh) : static_cast<int>(blockIdx.x);
  const int sub = cta / bh;
  const int b = (cta % bh) / args.Hkv;
  const int g = cta % args.Hkv;

  // Absolute position of query row 0, the sub-chunk's rows [r0, r1) and the
  // key range of the sequence (keys at or beyond seq_kv are never used).
  int pos0 = args.start;
  int Lb = args.L;                                      // query rows of this sequence (args.L is the row stride)
  if (args.ctx_lens != nullptr) {
    const int ctx = args.ctx_lens[b];
    if (ctx < args.L || ctx > args.max_ctx) {
      if (threadIdx.x == 0) atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
      return;
    }
    pos0 = ctx - args.L;
  }
  if (args.starts != nullptr) {
    pos0 = args.starts[b];
    Lb = args.lens[b];
    if (pos0 < 0 || Lb < 0 || Lb > args.L || pos0 + Lb > args.max_ctx) {
      if (threadIdx.x == 0) atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
      return;
    }
    if (Lb == 0) return;
  }
  const int seq_kv = pos0 + Lb;
  const int split = min(Lb, (pos0 / kTileKeys + 1) * kTileKeys - pos0);   // rows before the first tile boundary
  const int r0 = (sub == 0) ? 0 : split;
  const int r1 = (sub == 0) ? split : Lb;
  const int Lc = r1 - r0;
  if (Lc <= 0) return;                                  // the chunk does not reach a second tile
  const int n_rows = kGroup * Lc;                       // packed rows in use
  const int n_kv = (pos0 + r1 - 1) / kTileKeys + 1;     // C1: KV tiles 0..floor(last position / 128)
  // the tiles this CTA runs: all of them, or one C5 segment
  int j0 = 0, j1 = n_kv;
  if (args.seg_tiles > 0) {
    j0 = seg * args.seg_tiles;
    if (j0 >= n_kv) return;                             // the rows end before this segment
    j1 = min(n_kv, j0 + args.seg_tiles);
  }
  const int nt = j1 - j0;
  const bool has_last = (j1 == n_kv);
  const bool zero_tail = (args.block_table != nullptr) || (args.ctx_lens != nullptr) || (args.starts != nullptr);
  const int tail_from = seq_kv - (n_kv - 1) * kTileKeys;   // first V row of the last tile past the sequence

  // Q: packed row m = head i * Lc + rr holds q[b, 4g+i, r0+rr]; unused rows
  // are zero.  Written in the 128-byte swizzled layout the MMA descriptor
  // expects (16-byte chunk c of row m sits at chunk c ^ (m % 8)).
  for (int idx = threadIdx.x; idx < Cfg::kQRows * 16; idx += Cfg::kThreads) {
    const int m = idx >> 4;
    const int c = idx & 15;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (m < n_rows) {
      const int i = m / Lc;
      const int r = r0 + m % Lc;
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(args.q) +
          ((static_cast<size_t>(b) * args.Hq + g * kGroup + i) * args.L + r) * kHeadDim);
      val = __ldg(src + c);
    }
    *reinterpret_cast<uint4*>(smem + Cfg::kQOff + (c >> 3) * Cfg::kQSlab + (m >> 3) * 1024 + (m & 7) * 128 +
                              (((c & 7) ^ (m & 7)) << 4)) = val;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i)
      mbar_init(bar(i), (i >= Cfg::kBarPFull && i < Cfg::kBarPFull + Cfg::kSBufs)
                            ? static_cast<uint32_t>(32 * Cfg::kSoftmaxWarps) : 1u);
    misc[1] = (*reinterpret_cast<volatile uint32_t*>(args.err) != 0) ? 1u : 0u;
    fence_mbar_init();
  }
  fence_proxy_async_smem();   // generic-proxy Q writes -> visible to the tensor core
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(sbase + Cfg::kMiscOff, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const bool skip = (*abort_flag != 0);

  if (warp == Cfg::kProdWarp) {
    // ------------------------------------------------------------ producer
    if (!skip) {
      if (lane == 0) {
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
      }
      const uint64_t stream_once = l2_policy_evict_first();
      int issued = 0;
      bool ok = true;
      for (int jj = 0; jj < nt && ok; ++jj) {
        const int slot = jj % Cfg::kStages;
        const uint32_t use = jj / Cfg::kStages;
        int row = 0, plane = 0;
        if (lane == 0) kv_tile_coords(args, b, g, j0 + jj, row, plane);
        if (jj >= Cfg::kStages)
          ok = mbar_wait(bar(Cfg::kBarKEmpty + slot), (use - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t kdst = sbase + Cfg::kKOff + slot * kTileBytes;
          mbar_arrive_expect_tx(bar(Cfg::kBarKFull + slot), kTileBytes);
          tma_load_tile_hint(kdst, &tmap_k, row, plane, bar(Cfg::kBarKFull + slot), stream_once);
        }
        issued = 2 * jj + 1;
        if (jj >= Cfg::kStages)
          ok = mbar_wait(bar(Cfg::kBarVEmpty + slot), (use - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t vdst = sbase + Cfg::kVOff + slot * kTileBytes;
          mbar_arrive_expect_tx(bar(Cfg::kBarVFull + slot), kTileBytes);
          tma_load_tile_hint(vdst, &tmap_v, row, plane, bar(Cfg::kBarVFull + slot), stream_once);
        }
        issued = 2 * jj + 2;
      }
      if (ok && zero_tail && has_last) {
        // V rows past the sequence in its last tile may hold anything (another
        // sequence's data, NaN): make them zero so P = 0 contributes nothing.
        const int jl = nt - 1;
        const int slot = jl % Cfg::kStages;
        ok = mbar_wait(bar(Cfg::kBarVFull + slot), (jl / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          uint8_t* vt = smem + Cfg::kVOff + slot * kTileBytes;
          for (int idx = tail_from * 16 + lane; idx < kTileKeys * 16; idx += 32) {
            const int row = idx >> 4;
            const int c = idx & 15;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kSlabBytes + (row >> 3) * 1024 + (row & 7) * 128 +
                                      (((c & 7) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(Cfg::kBarVReady));
        }
      }
      if (!ok && lane == 0) {
        for (int x = (issued > 2 * Cfg::kStages ? issued - 2 * Cfg::kStages : 0); x < issued; ++x) {
          const int j = x >> 1;
          packed_drain_wait(bar(((x & 1) ? Cfg::kBarVFull : Cfg::kBarKFull) + j % Cfg::kStages),
                            (j / Cfg::kStages) & 1);
        }
      }
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && !skip) {
      const uint32_t q_saddr = sbase + Cfg::kQOff;
      bool ok = mbar_wait(bar(Cfg::kBarKFull), 0, abort_flag, args.err, kDevTimeoutTma);
      if (ok) {
        tc_fence_after();
        issue_qk(tmem_base, q_saddr, Cfg::kQSbo, Cfg::kQSlab, sbase + Cfg::kKOff);
        tc_commit(bar(Cfg::kBarSFull));
        tc_commit(bar(Cfg::kBarKEmpty));
      }
      for (int j = 0; j < nt && ok; ++j) {                  // j: tile j0 + j, ring and buffer index
        if (j + 1 < nt) {
          const int jn = j + 1;
          const int slot = jn % Cfg::kStages;
          ok = mbar_wait(bar(Cfg::kBarKFull + slot), (jn / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
          // S buffer jn%3 held P of tile jn-3: free once that P V has finished
          const int sb = jn % Cfg::kSBufs;
          if (ok && jn >= Cfg::kSBufs)
            ok = mbar_wait(bar(Cfg::kBarOFull + sb), ((jn - Cfg::kSBufs) / Cfg::kSBufs) & 1, abort_flag, args.err,
                           kDevTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          issue_qk(tmem_base + sb * 128u, q_saddr, Cfg::kQSbo, Cfg::kQSlab, sbase + Cfg::kKOff + slot * kTileBytes);
          tc_commit(bar(Cfg::kBarSFull + sb));
          tc_commit(bar(Cfg::kBarKEmpty + slot));
        }
        const int slot = j % Cfg::kStages;
        ok = mbar_wait(bar(Cfg::kBarPFull + j % Cfg::kSBufs), (j / Cfg::kSBufs) & 1, abort_flag, args.err,
                       kDevTimeoutSoftmax);
        if (ok) {
          if (zero_tail && has_last && j == nt - 1)
            ok = mbar_wait(bar(Cfg::kBarVReady), 0, abort_flag, args.err, kDevTimeoutTma);
          else
            ok = mbar_wait(bar(Cfg::kBarVFull + slot), (j / Cfg::kStages) & 1, abort_flag, args.err,
                           kDevTimeoutTma);
        }
        if (!ok) break;
        tc_fence_after();
        issue_pv(tmem_base + Cfg::kOCol, tmem_base + (j % Cfg::kSBufs) * 128u, sbase + Cfg::kVOff + slot * kTileBytes,
                 j == 0);                                   // the range's first tile clears O
        tc_commit(bar(Cfg::kBarOFull + j % Cfg::kSBufs));
        tc_commit(bar(Cfg::kBarVEmpty + slot));
      }
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain));
        packed_drain_wait(bar(Cfg::kBarDrain), 0);
      }
    }
  } else if (kWide) {
    // ------------------------------------------------- softmax, row per thread
    const int m = warp * 32 + lane;                    // packed row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t o_tmem = tmem_base + Cfg::kOCol + lane_off;
    const int head = (m < n_rows) ? m / Lc : 0;
    const int r = (m < n_rows) ? r0 + m % Lc : r0;     // unused rows take the sub-chunk's first position
    const int pos = pos0 + r;
    RowState st = row_state_init();
    bool ok = !skip;
    for (int j = 0; j < nt && ok; ++j) {                    // j: tile j0 + j
      ok = mbar_wait(bar(Cfg::kBarSFull + j % Cfg::kSBufs), (j / Cfg::kSBufs) & 1, abort_flag, args.err,
                     kDevTimeoutMma);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tmem = tmem_base + (j % Cfg::kSBufs) * 128u + lane_off;
      uint32_t s[128];
      tmem_ld128_wait(s_tmem, s);
      uint32_t p[64];
      const int jt = j0 + j;
      const float alpha = (jt == n_kv - 1) ? row_softmax_tile<true>(s, pos - jt * kTileKeys + 1, st, p)
                                           : row_softmax_tile<false>(s, kTileKeys, st, p);
      // O is rescaled only when some row's reference max moved, and only then
      // must the previous tile's P V have finished (its barrier is that tile's
      // S buffer's; the MMA issuer's wait before reusing an S buffer keeps it
      // at most one phase away).  P of this tile goes to its own S buffer, so
      // publishing it needs no wait.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        ok = mbar_wait(bar(Cfg::kBarOFull + (j - 1) % Cfg::kSBufs), ((j - 1) / Cfg::kSBufs) & 1, abort_flag,
                       args.err, kDevTimeoutMma);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(o_tmem + c * 32u, o);
          rescale32(o, alpha);
          tmem_st32(o_tmem + c * 32u, o);
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
      mbar_arrive(bar(Cfg::kBarPFull + j % Cfg::kSBufs));
    }
    if (ok)
      ok = mbar_wait(bar(Cfg::kBarOFull + (nt - 1) % Cfg::kSBufs), ((nt - 1) / Cfg::kSBufs) & 1, abort_flag,
                     args.err, kDevTimeoutMma);
    ok = __all_sync(0xffffffffu, ok);
    if (ok && args.part != nullptr) {
      // C5: this segment's partial (O unnormalised, m, mc, l) for the fold
      tc_fence_after();
      const bool store = m < n_rows;
      float* dst = args.part + ((((static_cast<size_t>(b) * args.Hq + g * kGroup + head) * args.L + r) * args.n_seg +
                                 seg) * kPartFloats);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32_wait(o_tmem + c * 32u, o);                // collective: every lane loads
        if (store) {
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            reinterpret_cast<float4*>(dst + 32 * c)[v4] =
                make_float4(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1]),
                            __uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3]));
        }
      }
      if (store) reinterpret_cast<float4*>(dst + 128)[0] = make_float4(st.m, st.mc, st.l, 0.0f);
    } else if (ok) {
      tc_fence_after();
      const float inv_l = row_inv_l(st);
      const bool store = m < n_rows;
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<__nv_bfloat16*>(args.o) +
          ((static_cast<size_t>(b) * args.Hq + g * kGroup + head) * args.L + r) * kHeadDim);
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
  } else {
    // ------------------------------------- softmax, four threads per row (narrow)
    // Rows 0..7 live in TMEM lanes 0..7; the 16x256b load gives each quad of
    // lanes 4i..4i+3 row i, thread u holding keys 8r+2u, 8r+2u+1 (r = 0..15),
    // so the row's 128 exponentials are spread over four threads.
    const int m = lane >> 2;                           // packed row 0..7
    const int u = lane & 3;
    const uint32_t o_tmem = tmem_base + Cfg::kOCol;    // warp 0: lanes 0..31
    const int head = (m < n_rows) ? m / Lc : 0;
    const int r = (m < n_rows) ? r0 + m % Lc : r0;     // unused rows take the sub-chunk's first position
    const int pos = pos0 + r;
    RowState st = row_state_init();
    bool ok = !skip;
    for (int j = 0; j < nt && ok; ++j) {                    // j: tile j0 + j
      ok = mbar_wait(bar(Cfg::kBarSFull + j % Cfg::kSBufs), (j / Cfg::kSBufs) & 1, abort_flag, args.err,
                     kDevTimeoutMma);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tmem = tmem_base + (j % Cfg::kSBufs) * 128u;
      float x[32];
      {
        uint32_t v0[32], v1[32];
        tmem_ld_16x256b_x8_pair_wait(s_tmem, s_tmem + 64u, v0, v1);   // keys 0..63, 64..127
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          x[2 * q] = __uint_as_float(v0[4 * q]);
          x[2 * q + 1] = __uint_as_float(v0[4 * q + 1]);
          x[16 + 2 * q] = __uint_as_float(v1[4 * q]);
          x[16 + 2 * q + 1] = __uint_as_float(v1[4 * q + 1]);
        }
      }
      uint32_t p[16];
      const int jt = j0 + j;
      const float alpha = (jt == n_kv - 1) ? row_softmax_tile_quad<true>(x, u, pos - jt * kTileKeys + 1, st, p)
                                           : row_softmax_tile_quad<false>(x, u, kTileKeys, st, p);
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        // rescale O (rows in lanes 0..31 through the 32x32b shape; lane L takes
        // the factor of row L % 8, rows 8..31 are never stored)
        ok = mbar_wait(bar(Cfg::kBarOFull + (j - 1) % Cfg::kSBufs), ((j - 1) / Cfg::kSBufs) & 1, abort_flag,
                       args.err, kDevTimeoutMma);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float a_lane = __shfl_sync(0xffffffffu, alpha, 4 * (lane & 7));
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(o_tmem + c * 32u, o);
          rescale32(o, a_lane);
          tmem_st32(o_tmem + c * 32u, o);
        }
      }
      {
        uint32_t pv[32];
#pragma unroll
        for (int q = 0; q < 16; ++q) { pv[2 * q] = p[q]; pv[2 * q + 1] = p[q]; }   // lanes m and m + 8
        tmem_st_16x128b_x16(s_tmem, pv);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Cfg::kBarPFull + j % Cfg::kSBufs));
    }
    if (ok)
      ok = mbar_wait(bar(Cfg::kBarOFull + (nt - 1) % Cfg::kSBufs), ((nt - 1) / Cfg::kSBufs) & 1, abort_flag,
                     args.err, kDevTimeoutMma);
    ok = __all_sync(0xffffffffu, ok);
    if (ok && args.part != nullptr) {
      // C5: lane L < 8 writes row L's partial; the state comes from its quad
      tc_fence_after();
      const float m_lane = __shfl_sync(0xffffffffu, st.m, 4 * (lane & 7));
      const float mc_lane = __shfl_sync(0xffffffffu, st.mc, 4 * (lane & 7));
      const float l_lane = __shfl_sync(0xffffffffu, st.l, 4 * (lane & 7));
      const int row = lane;
      const bool store = row < n_rows;
      const int s_head = store ? row / Lc : 0;
      const int s_r = store ? r0 + row % Lc : r0;
      float* dst = args.part + ((((static_cast<size_t>(b) * args.Hq + g * kGroup + s_head) * args.L + s_r) *
                                 args.n_seg + seg) * kPartFloats);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32_wait(o_tmem + c * 32u, o);
        if (store) {
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            reinterpret_cast<float4*>(dst + 32 * c)[v4] =
                make_float4(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1]),
                            __uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3]));
        }
      }
      if (store) reinterpret_cast<float4*>(dst + 128)[0] = make_float4(m_lane, mc_lane, l_lane, 0.0f);
    } else if (ok) {
      tc_fence_after();
      // lane L < 8 stores row L; its l comes from the quad that owns the row
      const float l_lane = __shfl_sync(0xffffffffu, st.l, 4 * (lane & 7));
      const float inv_l = __frcp_rn(l_lane);
      const int row = lane;
      const bool store = row < n_rows;
      const int s_head = store ? row / Lc : 0;
      const int s_r = store ? r0 + row % Lc : r0;
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<__nv_bfloat16*>(args.o) +
          ((static_cast<size_t>(b) * args.Hq + g * kGroup + s_head) * args.L + s_r) * kHeadDim);
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

template <bool kWide>
static cudaError_t launch_packed_t(const CUtensorMap& tk, const CUtensorMap& tv, const PackedArgs& a, int n_sub,
                                   cudaStream_t s) {
  using Cfg = PackedCfg<kWide>;
  static_assert(Cfg::kSmemUsed <= 227u * 1024u, "shared memory budget");
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kb_decode_kernel<kWide>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const unsigned grid = static_cast<unsigned>((a.seg_tiles > 0 ? a.n_seg : 1) * n_sub * a.B * a.Hkv);
  kb_decode_kernel<kWide><<<grid, Cfg::kThreads, Cfg::kSmemBytes, s>>>(tk, tv, a);
  return cudaGetLastError();
}

cudaError_t launch_packed(const CUtensorMap& tk, const CUtensorMap& tv, const PackedArgs& a, int n_sub,
                          cudaStream_t s) {
  // narrow when at most 8 rows are packed (two query rows per head)
  if (a.L <= 2) return launch_packed_t<false>(tk, tv, a, n_sub, s);
  return launch_packed_t<true>(tk, tv, a, n_sub, s);
}

// A kernel that waits on an mbarrier nobody ever signals, with a short limit:
// it exercises the bounded-wait path (error word set, kernel returns) without
// hanging or faulting the GPU.
__global__ void kb_wait_probe_kernel(uint32_t* err, unsigned long long limit_ns) {
  __shared__ uint64_t barrier_word;
  __shared__ uint32_t abort_word;
  const uint32_t b = smem_addr(&barrier_word);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(b, 0, &abort_word, err, kDevTimeoutProbe, limit_ns);
}

cudaError_t launch_wait_probe(uint32_t* err, unsigned long long limit_ns, cudaStream_t s) {
  kb_wait_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace kb
