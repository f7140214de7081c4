// kb_prefill2.cu -- causal GQA forward for a block of query rows against a KV
// cache (prefill and partitioned forward), one 128-row query tile per CTA
// with three S buffers in TMEM, so Q K^T of the next KV tiles runs on the
// tensor core while the softmax of the current one runs on the SM
// (KernelBraid README, "Method": GPU-specific tiling, data movement and
// parallelism are optimised within the numerical contract).
//
// The softmax of a row is spread over a quad of four threads through the
// 16x256b TMEM load (thread u holds keys 8r+2u, 8r+2u+1 of every group of 8,
// exactly the keys of the contract's partial sums k mod 8 = 2u, 2u+1), so the
// row math is the contract's, bit for bit (row_softmax_tile_quad).
//   warps 0..7   softmax: warp w owns TMEM lanes 32(w%4) + 16(w/4) .. +15;
//                thread t of it rows lane t/4 and lane t/4 + 8 of that block
//   warp 8       TMA producer of Q and the K ring (lane 0 issues)
//   warp 9       TMEM allocator + Q K^T issuer (one lane)
//   warp 10      TMA producer of the V ring (the warp zeroes a V tail)
//   warp 11      P V issuer (one lane)
//   warps 12..15 fold and epilogue: thread t of warp 12+i owns row 32i+t
// TMEM: S0 [0,128), S1 [128,256), S2 [256,384), O [384,512); P of a tile
// overwrites the first 64 columns of its S buffer.
//
// Segments (contract C5).  O in TMEM accumulates the running segment only.
// When a segment ends, the softmax warps leave its rows' (m, l) in shared
// memory and go on with the next tile; the fold warpgroup reads the
// segment's O once its last P V is done, which lets the P V issuer clear O
// for the next segment, and folds it into the row's folded O, held in its
// own registers (128 per thread; setmaxnreg moves registers from the
// producer/issuer warps to it).  After a unit's last segment the fold warps
// normalise and store the rows, so the softmax warps never wait for O.
#include "kb_contract.cuh"
#include "kb_launch.h"

namespace kb {

struct Prefill2Cfg {
  static constexpr int kThreads = 512;
  static constexpr int kLoadWarpK = 8;
  static constexpr int kMmaWarp = 9;                        // TMEM allocator + Q K^T issuer
  static constexpr int kLoadWarpV = 10;
  static constexpr int kPvWarp = 11;                        // P V issuer
  static constexpr int kFoldWarp0 = 12;                     // warps 12..15: fold and epilogue
  static constexpr int kStages = 3;
  static constexpr int kSBufs = kStages;                    // K slot j%3 frees when S(j) lands
  static constexpr uint32_t kTmemCols = 512;                // S0, S1, S2, O
  static constexpr uint32_t kOCol = kSBufs * 128u;          // O of the running segment
  // registers per thread after setmaxnreg: the 512 x 128 registers of the
  // launch split between 256 softmax, 128 producer/issuer and 128 fold threads
  static constexpr uint32_t kSoftmaxRegs = 136;
  static constexpr uint32_t kOtherRegs = 64;
  static constexpr uint32_t kFoldRegs = 176;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = kTileBytes;
  static constexpr uint32_t kVOff = kKOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 1;
  static constexpr int kBarVFull = kBarKFull + kStages;
  // per S buffer j%3: S(j) written (also: K slot j%3 free), P(j) written
  // (256 arrivals), P V(j) finished (also: V slot j%3 free)
  static constexpr int kBarSFull = kBarVFull + kStages;
  static constexpr int kBarPFull = kBarSFull + kSBufs;
  static constexpr int kBarOFull = kBarPFull + kSBufs;
  // per V slot: a unit's last V tile landed there with its tail zeroed
  static constexpr int kBarVReady = kBarOFull + kSBufs;
  static constexpr int kBarQEmpty = kBarVReady + kStages;  // a unit's last Q K^T done: Q may be replaced
  static constexpr int kBarORead = kBarQEmpty + 1;         // a finished segment's O was read (128 fold threads)
  static constexpr int kBarStFull = kBarORead + 1;         // a finished segment's (m, l) written (256 softmax)
  static constexpr int kBarStEmpty = kBarStFull + 1;       // ... and read (128 fold threads)
  static constexpr int kBarDrain = kBarStEmpty + 1;        // 2: one per MMA issuer
  static constexpr int kNumBars = kBarDrain + 2;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStatsOff = kMiscOff + 16;      // float2 (m, l) per row
  static constexpr uint32_t kSmemUsed = kStatsOff + kTileRows * 8;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
};
static_assert(8 * 32 * Prefill2Cfg::kSoftmaxRegs + 4 * 32 * Prefill2Cfg::kOtherRegs + 4 * 32 * Prefill2Cfg::kFoldRegs <=
                  512 * 128,
              "register split above the launch's registers");

__device__ __forceinline__ void drain_wait2(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 50000000ull) break;
}

// One work unit: (b, head, absolute query tile) and its geometry.
// Persistent launch with pairs (one CTA per SM): units come in pairs of one
// head's query-tile ranks r and n-1-r, whose causal lengths add up to n+1 key
// tiles whatever r is; a CTA runs pairs blockIdx.x, blockIdx.x + gridDim.x,
// ..., so every CTA gets the same work to within one pair.  Pairs are
// numbered (b, kv head) slowest, so the CTAs resident at one time share one
// GQA group's K/V in L2.
// Persistent launch with a snake: single units, longest first (query-tile
// rank slowest, then b and head), dealt to the CTAs 0..G-1 at even steps and
// G-1..0 at odd ones, which balances to within a few key tiles when a CTA
// gets only a few pairs' worth of work; every group's K/V is in use at once,
// so the host takes it only when all of K and V fit in L2 with room.
// Otherwise: one unit per CTA, longest first (the hardware scheduler
// balances), group-major or query-tile-major.
struct Unit {
  int b, g, h, t;       // batch, kv head, query head, absolute query tile
  int start, L;         // the sequence's first query position and row count
  int n_kv;             // C1: key tiles 0..t
  bool zero_tail;       // the last V tile's rows past the sequence are zeroed
  int kv_len;
};

__device__ __forceinline__ int pairs_per_group(const PrefillArgs& args) {
  return ((args.n_tiles + 1) / 2) * kGroup;
}

// Unit `second` (0: rank r, 1: rank n-1-r) of pair p.  False when that unit
// does not exist (the middle rank of an odd n, or a ragged batch's shorter
// sequence); a bad per-sequence start or length is reported and skipped.
__device__ __forceinline__ bool unit_of(int p, int second, const PrefillArgs& args, Unit& w) {
  int tile_rank;
  if (args.persistent == kSchedPairs) {
    const int ppg = pairs_per_group(args);
    const int bg = p / ppg;
    const int rem = p % ppg;
    const int r = rem / kGroup;
    tile_rank = second ? args.n_tiles - 1 - r : r;
    if (second && tile_rank == r) return false;
    w.b = bg / args.Hkv;
    w.g = bg % args.Hkv;
    w.h = w.g * kGroup + rem % kGroup;
  } else if (args.persistent == kSchedOnePerCta && args.group_major) {
    const int units_per_group = args.n_tiles * kGroup;
    const int bg = p / units_per_group;
    const int rem = p % units_per_group;
    tile_rank = rem / kGroup;
    w.b = bg / args.Hkv;
    w.g = bg % args.Hkv;
    w.h = w.g * kGroup + rem % kGroup;
  } else {
    tile_rank = p / (args.B * args.Hq);
    const int rem = p % (args.B * args.Hq);
    w.b = rem / args.Hq;
    w.h = rem % args.Hq;
    w.g = w.h / kGroup;
  }
  int first_tile = args.first_tile, n_tiles = args.n_tiles;
  w.start = args.start;
  w.L = args.L;
  if (args.starts != nullptr) {
    w.start = args.starts[w.b];
    w.L = args.lens[w.b];
    if (w.start < 0 || w.L < 0 || w.L > args.L || w.start + w.L > args.kv_cap) {
      if (threadIdx.x == 0 && tile_rank == 0 && (w.h % kGroup) == 0)
        atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
      return false;
    }
    if (w.L == 0) return false;
    first_tile = w.start / kTileRows;
    n_tiles = (w.start + w.L - 1) / kTileRows - first_tile + 1;
  }
  if (tile_rank >= n_tiles) return false;
  w.t = first_tile + n_tiles - 1 - tile_rank;
  w.n_kv = w.t + 1;
  w.kv_len = w.start + w.L;
  w.zero_tail = (args.block_table != nullptr) || (args.starts != nullptr);
  return true;
}

// C5 fold of 16 columns of a segment's O into the folded O (columns base..).
__device__ __forceinline__ void fold_chunk(uint32_t (&oacc)[128], int base, const uint32_t (&o)[16], FoldScale f) {
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float2 r = fold_o2(make_float2(__uint_as_float(oacc[base + i]), __uint_as_float(oacc[base + i + 1])),
                             make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f);
    oacc[base + i] = __float_as_uint(r.x);
    oacc[base + i + 1] = __float_as_uint(r.y);
  }
}

// The item a CTA runs at its step k: blockIdx.x + k * gridDim.x, or for the
// snake every odd step from the other end.
__device__ __forceinline__ int item_at(int k, const PrefillArgs& args) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return k * G + ((args.persistent == kSchedSnake && (k & 1)) ? G - 1 - c : c);
}

// Every role of a CTA walks the same units in the same order.
#define KB_FOR_EACH_UNIT(w)                                                                       \
  for (int kb_k = 0, kb_p = item_at(0, args); kb_p < n_items; ++kb_k, kb_p = item_at(kb_k, args)) \
    for (int kb_second = 0; kb_second < (args.persistent == kSchedPairs ? 2 : 1); ++kb_second)     \
      if (Unit w; unit_of(kb_p, kb_second, args, w))

__global__ void __launch_bounds__(Prefill2Cfg::kThreads, 1)
kb_prefill_kernel_s2(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs args) {
  using Cfg = Prefill2Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) { return smem_addr(bars + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = args.persistent == kSchedPairs ? args.B * args.Hkv * pairs_per_group(args)   // pairs
                                                     : args.n_tiles * args.B * args.Hq;            // units
  // C5 segment length in key tiles (0: the whole row is one segment)
  const int seg = args.seg_tiles > 0 ? args.seg_tiles : 0x40000000;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i) {
      uint32_t count = 1u;
      if ((i >= Cfg::kBarPFull && i < Cfg::kBarPFull + Cfg::kSBufs) || i == Cfg::kBarStFull) count = 256u;
      if (i == Cfg::kBarORead || i == Cfg::kBarStEmpty) count = 128u;
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
  // Every role walks the same units and counts the tiles it has handled (T)
  // and the units (U); ring slots, S buffers and every barrier parity follow
  // from those counts, so the CTA's units form one continuous pipeline.

  if (warp >= Cfg::kFoldWarp0) {
    // ------------------------------------------------- fold and epilogue
    // Walks the same units; per segment: wait for its (m, l) from the
    // softmax warps and for its last P V, read O (then the next segment may
    // clear it), fold (C5) into the row's folded O in registers; after the
    // unit's last segment normalise (C4) and store the row.
    regs_increase<Cfg::kFoldRegs>();
    const int fw = warp - Cfg::kFoldWarp0;
    const int row = 32 * fw + lane;                                  // TMEM lane = query row of the tile
    const uint32_t o_tmem = tmem_base + Cfg::kOCol + (static_cast<uint32_t>(32 * fw) << 16);
    const float2* stats = reinterpret_cast<const float2*>(smem + Cfg::kStatsOff);
    const float c = score_scale_log2();
    int T = 0, G = 0;                                                // tiles, segments
    bool ok = !skip;
    KB_FOR_EACH_UNIT(w) {
      if (!ok) break;
      RowState acc = row_state_init();
      uint32_t oacc[128];
      for (int j = 0; j < w.n_kv && ok; j += seg, ++G) {
        const int t_last = T + min(w.n_kv, j + seg) - 1;             // the segment's last tile
        // the stats come first: they are written after P(t_last), so P V(t_last - 3) is done and the
        // wait on P V(t_last) below is within one phase of its barrier
        ok = mbar_wait_idle(bar(Cfg::kBarStFull), G & 1, abort_flag, args.err, kDevTimeoutSoftmax, 256);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const float2 st = stats[row];
        const RowState sg{st.x, __fmul_rn(st.x, c), st.y};
        mbar_arrive(bar(Cfg::kBarStEmpty));
        ok = mbar_wait_idle(bar(Cfg::kBarOFull + t_last % Cfg::kSBufs), (t_last / Cfg::kSBufs) & 1, abort_flag,
                            args.err, kDevTimeoutMma, 32);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (j == 0) {
          tmem_ld128_wait(o_tmem, oacc);                            // the first segment as it is
          acc = sg;
        } else {
          const FoldScale f = fold_state(acc, sg);
          // the load of chunk q+1 is in flight while chunk q is folded
          uint32_t oa[16], ob[16];
          tmem_ld16_issue(o_tmem, oa);
#pragma unroll
          for (int q = 0; q < 8; q += 2) {
            tmem_ld16_wait_for(oa);
            tmem_ld16_issue(o_tmem + 16u * (q + 1), ob);
            fold_chunk(oacc, 16 * q, oa, f);
            tmem_ld16_wait_for(ob);
            if (q + 2 < 8) tmem_ld16_issue(o_tmem + 16u * (q + 2), oa);
            fold_chunk(oacc, 16 * (q + 1), ob, f);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(Cfg::kBarORead));
      }
      T += w.n_kv;
      if (!ok) break;
      const int i = w.t * kTileRows + row - w.start;                 // query row index in q / o
      if (i >= 0 && i < w.L) {
        const float inv_l = row_inv_l(acc);
        if (args.lse != nullptr) {
          // natural-log log-sum-exp of the row's scaled scores: the weights are
          // 2^(s c - mc), so log2 sum_j 2^(s_j c) = mc + log2(l)
          constexpr float kLn2 = 0.69314718055994531f;
          args.lse[(static_cast<size_t>(w.b) * args.Hq + w.h) * static_cast<size_t>(args.L) + i] =
              __fmul_rn(__fadd_rn(acc.mc, log2f(acc.l)), kLn2);
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) +
                                              ((static_cast<size_t>(w.b) * args.Hq + w.h) * args.L + i) * kHeadDim);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wv[e] = pack_bf16x2(__fmul_rn(__uint_as_float(oacc[8 * q + 2 * e]), inv_l),
                                __fmul_rn(__uint_as_float(oacc[8 * q + 2 * e + 1]), inv_l));
          dst[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
  } else if (warp >= Cfg::kLoadWarpK) {
    regs_decrease<Cfg::kOtherRegs>();
    if (warp == Cfg::kLoadWarpK || warp == Cfg::kLoadWarpV) {
      // --------------------------------------------------------- producers
      // One warp per ring (Q and K; V with the tail zeroing): each ring runs
      // kStages tiles ahead of its consumer, across unit boundaries.
      const bool is_v = (warp == Cfg::kLoadWarpV);
      if (!skip) {
        const uint64_t keep = l2_policy_evict_last();
        const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
        const int full0 = is_v ? Cfg::kBarVFull : Cfg::kBarKFull;
        const int empty0 = is_v ? Cfg::kBarOFull : Cfg::kBarSFull;   // slot T%3 free: P V(T) / Q K^T(T) done
        const uint32_t ring = sbase + (is_v ? Cfg::kVOff : Cfg::kKOff);
        if (lane == 0) {
          tma_prefetch_desc(tmap);
          if (!is_v) tma_prefetch_desc(&tmap_q);
        }
        int T = 0, U = 0, q_loads = 0;
        bool ok = true;
        KB_FOR_EACH_UNIT(w) {
          if (!ok) break;
          const bool paged = args.block_table != nullptr;
          if (!is_v) {
            if (U > 0) ok = mbar_wait(bar(Cfg::kBarQEmpty), (U - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(bar(Cfg::kBarQFull), kTileBytes);
              tma_load_tile(sbase + Cfg::kQOff, &tmap_q, w.t * kTileRows - w.start, w.b * args.Hq + w.h,
                            bar(Cfg::kBarQFull));
            }
            ++q_loads;
          }
          for (int j = 0; j < w.n_kv; ++j, ++T) {
            const int slot = T % Cfg::kStages;
            int row = j * kTileKeys, plane = w.b * args.Hkv + w.g;
            if (paged && lane == 0) {
              int pg = args.block_table[static_cast<size_t>(w.b) * args.pages_per_seq + row / args.page_size];
              if (pg < 0 || pg >= args.num_pages) {
                atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
                pg = args.num_pages;       // beyond the map: the TMA unit reads zeros
              }
              row = row % args.page_size;
              plane = pg * args.Hkv + w.g;
            }
            if (T >= Cfg::kStages)
              ok = mbar_wait(bar(empty0 + slot), ((T / Cfg::kStages) - 1) & 1, abort_flag, args.err,
                             kDevTimeoutSlot);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(bar(full0 + slot), kTileBytes);
              tma_load_tile_hint(ring + slot * kTileBytes, tmap, row, plane, bar(full0 + slot), keep);
            }
          }
          if (ok && is_v && w.zero_tail) {
            // V rows past kv_len in the unit's last tile may hold anything: zero them
            const int TL = T - 1;
            const int slot = TL % Cfg::kStages;
            ok = mbar_wait(bar(Cfg::kBarVFull + slot), (TL / Cfg::kStages) & 1, abort_flag, args.err,
                           kDevTimeoutTma);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
              uint8_t* vt = smem + Cfg::kVOff + slot * kTileBytes;
              const int tail_from = min(kTileKeys, w.kv_len - (w.n_kv - 1) * kTileKeys);
              for (int idx = tail_from * 16 + lane; idx < kTileKeys * 16; idx += 32) {
                const int vr = idx >> 4;
                const int c = idx & 15;
                *reinterpret_cast<uint4*>(vt + (c >> 3) * kSlabBytes + (vr >> 3) * 1024 + (vr & 7) * 128 +
                                          (((c & 7) ^ (vr & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(Cfg::kBarVReady + slot));
            }
          }
          ++U;
        }
        if (!ok && lane == 0) {
          if (!is_v && q_loads > 0) drain_wait2(bar(Cfg::kBarQFull), (q_loads - 1) & 1);
          for (int x = (T > Cfg::kStages ? T - Cfg::kStages : 0); x < T; ++x)
            drain_wait2(bar(full0 + x % Cfg::kStages), (x / Cfg::kStages) & 1);
        }
      }
    } else if (warp == Cfg::kMmaWarp) {
      // ------------------------------------------------------ Q K^T issuer
      // S(T) goes to buffer T%3 once P V(T-3) has read P(T-3) there.  A
      // second thread issues P V, so that the tensor pipe always has the
      // other stream's instructions while one issuer waits on a barrier.
      // After a unit's last Q K^T the Q buffer is released for the next unit.
      if (lane == 0 && !skip) {
        const uint32_t q_saddr = sbase + Cfg::kQOff;
        int T = 0, U = 0;
        bool ok = true;
        KB_FOR_EACH_UNIT(w) {
          if (!ok) break;
          ok = mbar_wait(bar(Cfg::kBarQFull), U & 1, abort_flag, args.err, kDevTimeoutTma);
          for (int j = 0; j < w.n_kv && ok; ++j, ++T) {
            const int sb = T % Cfg::kSBufs;
            const uint32_t use = T / Cfg::kSBufs;
            ok = mbar_wait(bar(Cfg::kBarKFull + sb), use & 1, abort_flag, args.err, kDevTimeoutTma);
            if (ok && T >= Cfg::kSBufs)
              ok = mbar_wait(bar(Cfg::kBarOFull + sb), (use - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
            if (!ok) break;
            tc_fence_after();
            issue_qk(tmem_base + sb * 128u, q_saddr, 1024u, kSlabBytes, sbase + Cfg::kKOff + sb * kTileBytes);
            tc_commit(bar(Cfg::kBarSFull + sb));
          }
          if (ok) tc_commit(bar(Cfg::kBarQEmpty));
          ++U;
        }
        if (!ok) {
          tc_commit(bar(Cfg::kBarDrain));
          drain_wait2(bar(Cfg::kBarDrain), 0);
        }
      }
    } else {
      // -------------------------------------------------------- P V issuer
      // The first P V of every segment clears O, so it waits until the
      // fold warps have read the previous segment's O (the "O read"
      // barrier completes once per segment, in order).
      if (lane == 0 && !skip) {
        int T = 0, F = 0;                                           // F: segments started
        uint32_t zero_parity = 0;                                   // bit s: zero-tail phases of V slot s, mod 2
        bool ok = true;
        KB_FOR_EACH_UNIT(w) {
          if (!ok) break;
          int js = 0;                                               // tile index within its segment
          for (int j = 0; j < w.n_kv && ok; ++j, ++T) {
            const int sb = T % Cfg::kSBufs;
            const uint32_t use = T / Cfg::kSBufs;
            ok = mbar_wait_hint(bar(Cfg::kBarPFull + sb), use & 1, abort_flag, args.err, kDevTimeoutSoftmax);
            if (ok) {
              if (w.zero_tail && j == w.n_kv - 1) {
                ok = mbar_wait(bar(Cfg::kBarVReady + sb), (zero_parity >> sb) & 1u, abort_flag, args.err,
                               kDevTimeoutTma);
                zero_parity ^= 1u << sb;
              } else {
                ok = mbar_wait(bar(Cfg::kBarVFull + sb), use & 1, abort_flag, args.err, kDevTimeoutTma);
              }
            }
            const bool first = (js == 0);
            if (++js == seg) js = 0;
            if (ok && first && F > 0)
              ok = mbar_wait(bar(Cfg::kBarORead), (F - 1) & 1, abort_flag, args.err, kDevTimeoutSoftmax);
            if (!ok) break;
            tc_fence_after();
            issue_pv(tmem_base + Cfg::kOCol, tmem_base + sb * 128u, sbase + Cfg::kVOff + sb * kTileBytes, first);
            tc_commit(bar(Cfg::kBarOFull + sb));
            if (first) ++F;
          }
        }
        if (!ok) {
          tc_commit(bar(Cfg::kBarDrain + 1));
          drain_wait2(bar(Cfg::kBarDrain + 1), 0);
        }
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    regs_increase<Cfg::kSoftmaxRegs>();
    const int q4 = warp & 3;                                        // TMEM lane quarter of this warp
    const int lane_base = 32 * q4 + 16 * (warp >> 2);               // 16-lane block
    const uint32_t lane_off = static_cast<uint32_t>(lane_base) << 16;
    const int u = lane & 3;
    const int rA = lane_base + (lane >> 2);                         // rows (TMEM lanes) of this thread
    const int rB = rA + 8;
    const uint32_t o_tmem = tmem_base + Cfg::kOCol + lane_off;
    float2* stats = reinterpret_cast<float2*>(smem + Cfg::kStatsOff);
    int T = 0, G = 0;                                               // tiles, segments
    bool ok = !skip;
    KB_FOR_EACH_UNIT(w) {
      if (!ok) break;
      const int n_kv = w.n_kv;
      RowState sA = row_state_init(), sB = row_state_init();
      int js = 0;                                                   // tile index within its segment
      for (int j = 0; j < n_kv && ok; ++j, ++T) {
        const int sb = T % Cfg::kSBufs;
        ok = mbar_wait_hint(bar(Cfg::kBarSFull + sb), (T / Cfg::kSBufs) & 1, abort_flag, args.err, kDevTimeoutMma);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_tmem = tmem_base + sb * 128u + lane_off;
        float xA[32], xB[32];
        {
          uint32_t v0[32], v1[32];
          tmem_ld_16x256b_x8_pair_wait(s_tmem, s_tmem + 64u, v0, v1);   // keys 0..63, 64..127
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            xA[2 * r] = __uint_as_float(v0[4 * r]);
            xA[2 * r + 1] = __uint_as_float(v0[4 * r + 1]);
            xB[2 * r] = __uint_as_float(v0[4 * r + 2]);
            xB[2 * r + 1] = __uint_as_float(v0[4 * r + 3]);
            xA[16 + 2 * r] = __uint_as_float(v1[4 * r]);
            xA[16 + 2 * r + 1] = __uint_as_float(v1[4 * r + 1]);
            xB[16 + 2 * r] = __uint_as_float(v1[4 * r + 2]);
            xB[16 + 2 * r + 1] = __uint_as_float(v1[4 * r + 3]);
          }
        }
        const bool seg_start = (js == 0);
        if (++js == seg) js = 0;
        const bool seg_end = (js == 0) || (j == n_kv - 1);
        if (seg_start) {                                            // C5: each segment starts fresh
          sA = row_state_init();
          sB = row_state_init();
        }
        uint32_t pkA[16], pkB[16];
        float aA, aB;
        if (j == n_kv - 1) {                                        // diagonal tile: causal mask
          aA = row_softmax_tile_quad<true>(xA, u, rA + 1, sA, pkA);
          aB = row_softmax_tile_quad<true>(xB, u, rB + 1, sB, pkB);
        } else {
          aA = row_softmax_tile_quad<false>(xA, u, kTileKeys, sA, pkA);
          aB = row_softmax_tile_quad<false>(xB, u, kTileKeys, sB, pkB);
        }
        if (!seg_start && __any_sync(0xffffffffu, aA != 1.0f || aB != 1.0f)) {
          // O must hold P V of tile T-1 before it is rescaled; per-buffer
          // barriers keep this wait exact although it is only taken when
          // needed (P V(T-4) is done: S(T) was committed after it)
          ok = mbar_wait(bar(Cfg::kBarOFull + (T - 1) % Cfg::kSBufs), ((T - 1) / Cfg::kSBufs) & 1, abort_flag,
                         args.err, kDevTimeoutMma);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tmem_ld_16x256b_x8_wait(o_tmem + 64u * half, o);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const float2 ra = __fmul2_rn(make_float2(__uint_as_float(o[4 * r]), __uint_as_float(o[4 * r + 1])),
                                           make_float2(aA, aA));
              const float2 rb = __fmul2_rn(make_float2(__uint_as_float(o[4 * r + 2]), __uint_as_float(o[4 * r + 3])),
                                           make_float2(aB, aB));
              o[4 * r] = __float_as_uint(ra.x);
              o[4 * r + 1] = __float_as_uint(ra.y);
              o[4 * r + 2] = __float_as_uint(rb.x);
              o[4 * r + 3] = __float_as_uint(rb.y);
            }
            tmem_st_16x256b_x8(o_tmem + 64u * half, o);
          }
        }
        {
          uint32_t pv[32];
#pragma unroll
          for (int r = 0; r < 16; ++r) { pv[2 * r] = pkA[r]; pv[2 * r + 1] = pkB[r]; }
          tmem_st_16x128b_x16(s_tmem, pv);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(Cfg::kBarPFull + sb));
        if (seg_end) {
          // hand the finished segment's (m, l) to the fold warps, once they
          // have read the previous segment's
          if (G > 0) {
            ok = mbar_wait(bar(Cfg::kBarStEmpty), (G - 1) & 1, abort_flag, args.err, kDevTimeoutSoftmax);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
          }
          if (u == 0) {
            stats[rA] = make_float2(sA.m, sA.l);
            stats[rB] = make_float2(sB.m, sB.l);
          }
          mbar_arrive(bar(Cfg::kBarStFull));
          ++G;
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

cudaError_t launch_prefill_s2(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const PrefillArgs& a, cudaStream_t s) {
  using Cfg = Prefill2Cfg;
  static_assert(Cfg::kSmemBytes <= 227u * 1024u, "shared memory budget");
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kb_prefill_kernel_s2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // persistent: one CTA per SM at most, each walking its share of the unit
  // pairs or of the snake; otherwise one CTA per unit
  const long long pairs = static_cast<long long>((a.n_tiles + 1) / 2) * kGroup * a.B * a.Hkv;
  const long long units = static_cast<long long>(a.n_tiles) * a.B * a.Hq;
  const long long grid = a.persistent == kSchedPairs ? (pairs < a.max_ctas ? pairs : a.max_ctas)
                         : a.persistent == kSchedSnake ? (units < a.max_ctas ? units : a.max_ctas)
                                                       : units;
  kb_prefill_kernel_s2<<<static_cast<unsigned>(grid), Cfg::kThreads, Cfg::kSmemBytes, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace kb
