// kb_decode.cu -- query rows packed by GQA group: one-token decode (KernelBraid
// README, "Usage": unified_decode over the same KV context, whose output must
// equal the prefill row bit for bit; "Features": one query token per decode
// call) and chunks of up to 32 query rows against a KV cache (README
// "Method": partitioned forward execution), on a contiguous or a paged cache.
//
// The four query heads of the GQA group and the sub-chunk's rows are packed
// into the rows of the M=128 MMA (row m = head i * Lc + query row r), so the
// kernel issues the very same tcgen05.mma shape, k-order and row softmax as
// prefill and every packed row reproduces the prefill row exactly, while K
// and V are read once per KV head.  A sub-chunk never crosses a 128-position
// tile boundary, so all its rows end on the same KV tile.  K/V tiles stream
// through a three-deep TMA ring; S has three TMEM buffers (two in the wide fold mode),
// so the next Q K^T products run ahead of the softmax.
//   softmax        warps 0..NS-1 (NS = 1 narrow: a quad of threads per row,
//                  rows 0..7 in TMEM lanes 0..7; NS = 4 wide: a thread per row)
//   K producer     TMA loads of the K ring (lane 0 issues)
//   Q K^T issuer   TMEM allocator; one lane issues S(j) as soon as K(j) has
//                  landed and its S buffer is free
//   V producer     TMA loads of the V ring; the warp zeroes a V tail
//   P V issuer     one lane issues O += P(j) V(j) as soon as both are there
//   fold           narrow only, warp 4 (it reaches TMEM lanes 0..31, as warp
//                  0 does): segment folds and the epilogue
// Each ring and each product has its own thread, so a late K tile never holds
// back a P V (and with it the V slot the next V tile needs), nor the reverse.
// Narrow: warps 0 softmax, 1 K, 2 Q K^T, 3 V, 4 fold, 5 P V; wide: 0..3
// softmax, 4 K, 5 Q K^T, 6 V, 7 P V.
// Narrow (at most 8 packed rows): Q is one 8-row swizzle atom per d-slab and
// the row groups 8..127 of the MMA alias it (stride-byte-offset 0).
//
// Segments (contract C5), two ways:
//  - fold mode (the default entry points): the segments of a (sub-chunk,
//    batch, KV head) are split into contiguous blocks over a cluster of C
//    CTAs (C = 1 .. 8).  Each CTA runs its segments from the fresh state;
//    its softmax warp hands each finished segment's (m, l) to the fold warp,
//    which reads the segment's O.  The cluster's first CTA folds its own
//    segments as they finish, in registers.  The others write each segment's
//    partial (O, m, mc, l) into the first CTA's shared memory and arrive on
//    its barrier; the first CTA's fold warp writes its own folded segments
//    into the slot after them and arrives too, and warps 0-3 of that CTA
//    (their roles are over by then) fold the slots in segment order, 16
//    threads per row, and normalise.  When the partials do not fit there,
//    each CTA keeps its own until the first CTA has streamed its last tile,
//    then copies them into the first CTA's K/V rings in one bulk copy
//    ("gather"); past the rings' size (the longest contexts) the first CTA
//    reads them through distributed shared memory after a cluster barrier.
//    Narrow rows only take C > 1; wide chunks run C = 1 with the folded O in
//    TMEM.
//  - workspace mode (the *_seg entry points): one CTA per segment writes its
//    partial to a caller workspace, which kb_seg_fold_kernel folds.
#include "kb_contract.cuh"
#include "kb_launch.h"

namespace kb {

template <bool kWide, int kNumSBufs>
struct PackedCfg {
  static constexpr int kSoftmaxWarps = kWide ? 4 : 1;
  static constexpr int kKProdWarp = kWide ? 4 : 1;
  static constexpr int kQkWarp = kWide ? 5 : 2;             // TMEM allocator + Q K^T issuer
  static constexpr int kVProdWarp = kWide ? 6 : 3;
  static constexpr int kPvWarp = kWide ? 7 : 5;
  static constexpr int kFoldWarp = kWide ? -1 : 4;          // narrow: folds and epilogue
  static constexpr int kThreads = (kWide ? 8 : 6) * 32;
  static constexpr int kStages = 3;
  static constexpr int kQRows = kWide ? 128 : 8;
  static constexpr int kSBufs = kNumSBufs;
  static constexpr bool kFoldTmem = kWide && kNumSBufs == 2;  // wide fold mode: folded O in TMEM
  static constexpr uint32_t kTmemCols = 512;                  // S buffers, O (and the folded O)
  static constexpr uint32_t kOCol = kSBufs * 128u;
  static constexpr uint32_t kOAccCol = 384u;                  // kFoldTmem only
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
  static constexpr int kBarORead = kBarVReady + 1;         // a finished segment's O has been read
  static constexpr int kBarStFull = kBarORead + 1;         // narrow: a finished segment's (m, l) written
  static constexpr int kBarStEmpty = kBarStFull + 1;       // narrow: ... and read by the fold warp
  static constexpr int kBarPart = kBarStEmpty + 1;         // first CTA of a cluster: every partial written
  static constexpr int kBarDrain = kBarPart + 1;           // 2: one per MMA issuer
  static constexpr int kBarQReady = kBarDrain + 2;         // Q written to shared memory by its loaders
  static constexpr int kBarGo = kBarQReady + 1;            // gather: the first CTA's K/V rings are free
  static constexpr int kNumBars = kBarGo + 1;
  // Q is loaded by the softmax warps (and the fold warp when narrow) while
  // the producers' first K/V loads are already in flight
  static constexpr int kQLoaders = 32 * (kSoftmaxWarps + (kWide ? 0 : 1));
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStatsOff = kMiscOff + 16u;      // narrow: float2 (m, l) of rows 0..7
  // narrow: the rest of shared memory holds the segment partials a
  // non-first CTA of a cluster leaves for the first one
  static constexpr uint32_t kPartOff = (kStatsOff + 64u + 15u) & ~15u;
  static constexpr uint32_t kSmemCap = 227u * 1024u - 1024u;   // usable once the base is 1 KB aligned
  static constexpr uint32_t kPartBytes = kWide ? 0u : ((kSmemCap - kPartOff) & ~15u);
  static constexpr uint32_t kSmemUsed = kPartOff + kPartBytes;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
};

// Partials a narrow CTA can hold in shared memory, for n_rows packed rows.
uint32_t packed_partial_slots(int n_rows) {
  return PackedCfg<false, 3>::kPartBytes / (static_cast<uint32_t>(n_rows) * kPartFloats * 4u);
}

__device__ __forceinline__ void packed_drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 50000000ull) break;
}

// Row of the K/V tensor map and plane of key tile j of sequence b, KV head g.
// False for a page index out of range (reported; the coordinates then point
// beyond the map, where the TMA unit reads zeros).
__device__ __forceinline__ bool kv_tile_coords(const PackedArgs& a, int b, int g, int j, int& row, int& plane) {
  if (a.block_table == nullptr) {
    row = j * kTileKeys;
    plane = b * a.Hkv + g;
    return true;
  }
  const int key = j * kTileKeys;
  int pg = a.block_table[static_cast<size_t>(b) * a.pages_per_seq + key / a.page_size];
  bool ok = true;
  if (pg < 0 || pg >= a.num_pages) {
    atomicCAS(a.err, 0u, static_cast<uint32_t>(kDevBadInput));
    pg = a.num_pages;
    ok = false;
  }
  row = key % a.page_size;
  plane = pg * a.Hkv + g;
  return ok;
}

// First segment of cluster rank c when ns segments are cut into C contiguous
// blocks (ceil(c ns / C)): rank 0 always gets at least one segment.
__device__ __forceinline__ int seg_block_start(int c, int ns, int C) { return (c * ns + C - 1) / C; }

template <bool kWide, int kNumSBufs>
__global__ void __launch_bounds__(PackedCfg<kWide, kNumSBufs>::kThreads, 1)
kb_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const PackedArgs args) {
  using Cfg = PackedCfg<kWide, kNumSBufs>;
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
  const bool ws_mode = args.part != nullptr;                 // one segment per CTA, partials to a workspace
  const int C = ws_mode ? 1 : args.cluster;                  // CTAs per (sub-chunk, b, kv head)
  const int rank = ws_mode ? 0 : static_cast<int>(blockIdx.x) % C;
  const int seg_ws = ws_mode ? static_cast<int>(blockIdx.x) / (args.n_sub * bh) : 0;
  const int cta = ws_mode ? static_cast<int>(blockIdx.x) % (args.n_sub * bh) : static_cast<int>(blockIdx.x) / C;
  const int sub = cta / bh;
  const int b = (cta % bh) / args.Hkv;
  const int g = cta % args.Hkv;
  // No CTA returns early: a CTA of a cluster must reach the cluster barriers
  // below, so a CTA without work only skips its roles.
  bool active = true;

  // Absolute position of query row 0, the sub-chunk's rows [r0, r1) and the
  // key range of the sequence (keys at or beyond seq_kv are never used).
  int pos0 = args.start;
  int Lb = args.L;                                      // query rows of this sequence (args.L is the row stride)
  if (args.ctx_lens != nullptr) {
    const int ctx = args.ctx_lens[b];
    if (ctx < args.L || ctx > args.max_ctx) {
      if (threadIdx.x == 0) atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
      active = false;
    }
    pos0 = ctx - args.L;
  }
  if (args.starts != nullptr) {
    pos0 = args.starts[b];
    Lb = args.lens[b];
    if (pos0 < 0 || Lb < 0 || Lb > args.L || pos0 + Lb > args.max_ctx) {
      if (threadIdx.x == 0) atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
      active = false;
    }
    if (Lb == 0) active = false;
  }
  if (!active) {
    pos0 = 0;
    Lb = 1;
  }
  const int seq_kv = pos0 + Lb;
  const int split = min(Lb, (pos0 / kTileKeys + 1) * kTileKeys - pos0);   // rows before the first tile boundary
  const int r0 = (sub == 0) ? 0 : split;
  const int r1 = (sub == 0) ? split : Lb;
  const int Lc = max(r1 - r0, 1);
  if (r1 - r0 <= 0) active = false;                     // the chunk does not reach a second tile
  const int n_rows = kGroup * Lc;                       // packed rows in use
  const int n_kv = (pos0 + r1 - 1) / kTileKeys + 1;     // C1: KV tiles 0..floor(last position / 128)
  // the tiles this CTA runs: one C5 segment (workspace mode) or a contiguous
  // block of segments (fold mode)
  const int seg_len = ws_mode ? args.seg_tiles : args.fold_seg;
  const int ns = (n_kv + seg_len - 1) / seg_len;        // segments of the sub-chunk's rows
  int j0, j1;
  if (ws_mode) {
    j0 = seg_ws * seg_len;
    j1 = min(n_kv, j0 + seg_len);
  } else {
    j0 = seg_block_start(rank, ns, C) * seg_len;
    j1 = min(n_kv, seg_block_start(rank + 1, ns, C) * seg_len);
  }
  if (j0 >= j1) active = false;
  const int nt = active ? j1 - j0 : 0;
  const bool has_last = (j1 == n_kv);
  const bool zero_tail = (args.block_table != nullptr) || (args.ctx_lens != nullptr) || (args.starts != nullptr);
  const int tail_from = seq_kv - (n_kv - 1) * kTileKeys;   // first V row of the last tile past the sequence
  const uint32_t slot_bytes = static_cast<uint32_t>(n_rows) * kPartFloats * 4u;
  // fold mode, C > 1: the other CTAs' segments (from s_first on) reach the
  // first CTA's shared memory in one of three ways:
  //  - push: as each finishes, into the first CTA's partial slots, followed
  //    by the first CTA's own folded segments, when they all fit there;
  //  - gather: otherwise, when they fit in the first CTA's K/V rings: each
  //    CTA keeps its partials, and once the first CTA has streamed its last
  //    tile it lets the others copy them into its rings in one bulk copy each;
  //  - pull: otherwise (the longest contexts), the first CTA reads them from
  //    the others' shared memory after a cluster barrier.
  const int s_first = seg_block_start(1, ns, C);
  const bool push = C > 1 && !ws_mode &&
                    static_cast<uint32_t>(ns - s_first + 1) * slot_bytes <= static_cast<uint32_t>(Cfg::kPartBytes);
  const bool gather = !kWide && C > 1 && !ws_mode && !push &&
                      static_cast<uint32_t>(ns - s_first) * slot_bytes <= 2u * Cfg::kStages * kTileBytes;
  const bool pull_sync = C > 1 && !ws_mode && !push && !gather;   // the pull path's cluster barrier

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i) {
      uint32_t count = ((i >= Cfg::kBarPFull && i < Cfg::kBarPFull + Cfg::kSBufs) || i == Cfg::kBarORead ||
                        i == Cfg::kBarStFull || i == Cfg::kBarStEmpty)
                           ? static_cast<uint32_t>(32 * Cfg::kSoftmaxWarps) : 1u;
      // push: every fold warp of the cluster; gather: the first CTA's own
      // (the others' bytes complete its transaction count)
      if (i == Cfg::kBarPart && C > 1) count = static_cast<uint32_t>(push ? 32 * C : 32);
      if (i == Cfg::kBarQReady) count = static_cast<uint32_t>(Cfg::kQLoaders);
      mbar_init(bar(i), count);
    }
    misc[1] = 0u;
    if (gather && rank == 0) mbar_expect_tx(bar(Cfg::kBarPart), static_cast<uint32_t>(ns - s_first) * slot_bytes);
    fence_mbar_init();
  }
  if (warp == Cfg::kQkWarp) {
    tmem_alloc(sbase + Cfg::kMiscOff, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  // Nothing global is read before this point, so the producers' first loads
  // leave at once.  Each role reads the error word when it starts (the
  // producers once their first loads are in flight) and skips its work if
  // an earlier kernel recorded an error.
  const bool run = active;
  // every CTA of the cluster has initialised its barriers once this barrier
  // completes; its wait comes before any access to another CTA
  if (C > 1) cluster_arrive();

  const bool q_loader = warp < Cfg::kSoftmaxWarps || warp == Cfg::kFoldWarp;
  if (q_loader) {
    // Q: packed row m = head i * Lc + rr holds q[b, 4g+i, r0+rr]; unused rows
    // are zero.  Written in the 128-byte swizzled layout the MMA descriptor
    // expects (16-byte chunk c of row m sits at chunk c ^ (m % 8)).
    const int t = warp == Cfg::kFoldWarp ? 32 * Cfg::kSoftmaxWarps + lane : static_cast<int>(threadIdx.x);
    for (int idx = t; idx < Cfg::kQRows * 16; idx += Cfg::kQLoaders) {
      const int m = idx >> 4;
      const int c = idx & 15;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (active && m < n_rows) {
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
    fence_proxy_async_smem();   // generic-proxy Q writes -> visible to the tensor core
    mbar_arrive(bar(Cfg::kBarQReady));
  }

  if (warp == Cfg::kKProdWarp || warp == Cfg::kVProdWarp) {
    // ----------------------------------------------------------- producers
    // One warp per ring: a slot is refilled once its tile's product (Q K^T
    // for K, P V for V) has finished.
    const bool is_v = (warp == Cfg::kVProdWarp);
    if (run) {
      const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
      if (lane == 0) tma_prefetch_desc(tmap);
      const uint64_t stream_once = l2_policy_evict_first();
      const int full0 = is_v ? Cfg::kBarVFull : Cfg::kBarKFull;
      const int empty0 = is_v ? Cfg::kBarVEmpty : Cfg::kBarKEmpty;
      const uint32_t ring = sbase + (is_v ? Cfg::kVOff : Cfg::kKOff);
      int issued = 0;
      bool ok = true;
      for (int jj = 0; jj < nt && ok; ++jj) {
        const int slot = jj % Cfg::kStages;
        const uint32_t use = jj / Cfg::kStages;
        int row = 0, plane = 0;
        if (lane == 0) kv_tile_coords(args, b, g, j0 + jj, row, plane);
        if (jj == Cfg::kStages) ok = no_error(args.err, abort_flag);   // the first loads are in flight
        if (ok && jj >= Cfg::kStages)
          ok = mbar_wait(bar(empty0 + slot), (use - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(full0 + slot), kTileBytes);
          tma_load_tile_hint(ring + slot * kTileBytes, tmap, row, plane, bar(full0 + slot), stream_once);
        }
        issued = jj + 1;
      }
      if (ok && nt <= Cfg::kStages) ok = no_error(args.err, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok && is_v && zero_tail && has_last) {
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
        for (int x = (issued > Cfg::kStages ? issued - Cfg::kStages : 0); x < issued; ++x)
          packed_drain_wait(bar(full0 + x % Cfg::kStages), (x / Cfg::kStages) & 1);
      }
    }
    if (C > 1) {
      cluster_wait();
      if (pull_sync) cluster_sync();
    }
  } else if (warp == Cfg::kQkWarp) {
    // -------------------------------------------------------- Q K^T issuer
    // S(j) goes to buffer j%n once K(j) has landed and P V(j-n) has read
    // P(j-n) out of that buffer.
    if (lane == 0 && run) {
      const uint32_t q_saddr = sbase + Cfg::kQOff;
      bool ok = no_error(args.err, abort_flag) &&
                mbar_wait(bar(Cfg::kBarQReady), 0, abort_flag, args.err, kDevTimeoutTma);
      for (int j = 0; j < nt && ok; ++j) {                  // j: tile j0 + j
        const int slot = j % Cfg::kStages;
        const int sb = j % Cfg::kSBufs;
        ok = mbar_wait(bar(Cfg::kBarKFull + slot), (j / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        if (ok && j >= Cfg::kSBufs)
          ok = mbar_wait(bar(Cfg::kBarOFull + sb), ((j - Cfg::kSBufs) / Cfg::kSBufs) & 1, abort_flag, args.err,
                         kDevTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        issue_qk(tmem_base + sb * 128u, q_saddr, Cfg::kQSbo, Cfg::kQSlab, sbase + Cfg::kKOff + slot * kTileBytes);
        tc_commit(bar(Cfg::kBarSFull + sb));
        tc_commit(bar(Cfg::kBarKEmpty + slot));
      }
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain));
        packed_drain_wait(bar(Cfg::kBarDrain), 0);
      }
    }
    __syncwarp();
    if (C > 1) {
      cluster_wait();
      if (pull_sync) cluster_sync();
    }
  } else if (warp == Cfg::kPvWarp) {
    // ---------------------------------------------------------- P V issuer
    // The first P V of every segment clears O; after the CTA's first segment
    // it waits until the previous segment's O has been read.
    if (lane == 0 && run) {
      int F = 0;                                            // segments started
      int js = 0;                                           // tile index within its segment (j0 starts one)
      bool ok = no_error(args.err, abort_flag);
      for (int j = 0; j < nt && ok; ++j) {                  // j: tile j0 + j
        const int slot = j % Cfg::kStages;
        const int sb = j % Cfg::kSBufs;
        if (zero_tail && has_last && j == nt - 1)
          ok = mbar_wait(bar(Cfg::kBarVReady), 0, abort_flag, args.err, kDevTimeoutTma);
        else
          ok = mbar_wait(bar(Cfg::kBarVFull + slot), (j / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        const bool first = (js == 0);
        if (++js == seg_len) js = 0;
        if (ok && first && F > 0)
          ok = mbar_wait(bar(Cfg::kBarORead), (F - 1) & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (ok)
          ok = mbar_wait_hint(bar(Cfg::kBarPFull + sb), (j / Cfg::kSBufs) & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        issue_pv(tmem_base + Cfg::kOCol, tmem_base + sb * 128u, sbase + Cfg::kVOff + slot * kTileBytes, first);
        tc_commit(bar(Cfg::kBarOFull + sb));
        tc_commit(bar(Cfg::kBarVEmpty + slot));
        if (first) ++F;
      }
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain + 1));
        packed_drain_wait(bar(Cfg::kBarDrain + 1), 0);
      }
    }
    __syncwarp();
    if (C > 1) {
      cluster_wait();
      if (pull_sync) cluster_sync();
    }
  } else if constexpr (kWide) {
    // ------------------------------------------------- softmax, row per thread
    const int m = warp * 32 + lane;                    // packed row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t o_tmem = tmem_base + Cfg::kOCol + lane_off;
    const uint32_t oacc_tmem = tmem_base + Cfg::kOAccCol + lane_off;   // kFoldTmem only
    const int head = (m < n_rows) ? m / Lc : 0;
    const int r = (m < n_rows) ? r0 + m % Lc : r0;     // unused rows take the sub-chunk's first position
    const int pos = pos0 + r;
    RowState st = row_state_init(), prev = st, acc = st;
    int nfin = 0;                                      // segments finished (and folded into O_acc)
    int js = 0;                                        // tile index within its segment (j0 starts one)
    bool ok = run && no_error(args.err, abort_flag);
    for (int j = 0; j < nt && ok; ++j) {               // j: tile j0 + j
      ok = mbar_wait_hint(bar(Cfg::kBarSFull + j % Cfg::kSBufs), (j / Cfg::kSBufs) & 1, abort_flag, args.err,
                     kDevTimeoutMma);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tmem = tmem_base + (j % Cfg::kSBufs) * 128u + lane_off;
      uint32_t s[128];
      tmem_ld128_wait(s_tmem, s);
      uint32_t p[64];
      const int jt = j0 + j;
      const bool seg_start = (js == 0);
      if (++js == seg_len) js = 0;
      if (seg_start) {
        prev = st;
        st = row_state_init();
      }
      const float alpha = (jt == n_kv - 1) ? row_softmax_tile<true>(s, pos - jt * kTileKeys + 1, st, p)
                                           : row_softmax_tile<false>(s, kTileKeys, st, p);
      // O is rescaled only when some row's reference max moved, and only then
      // must the previous tile's P V have finished (its barrier is that tile's
      // S buffer's; the MMA issuer's wait before reusing an S buffer keeps it
      // at most one phase away).  P of this tile goes to its own S buffer, so
      // publishing it needs no wait.
      if (!seg_start && __any_sync(0xffffffffu, alpha != 1.0f)) {
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
      if constexpr (Cfg::kFoldTmem) {
        if (seg_start && j > 0) {
          // C5: fold the segment that ended with tile j-1 into O_acc (TMEM)
          ok = mbar_wait(bar(Cfg::kBarOFull + (j - 1) % Cfg::kSBufs), ((j - 1) / Cfg::kSBufs) & 1, abort_flag,
                         args.err, kDevTimeoutMma);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          FoldScale f{1.0f, 1.0f};
          if (nfin == 0) acc = prev;
          else f = fold_state(acc, prev);
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t os[32], oa[32];
            tmem_ld32_wait(o_tmem + c * 32u, os);
            if (nfin == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) oa[i] = os[i];
            } else {
              tmem_ld32_wait(oacc_tmem + c * 32u, oa);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 r2 = fold_o2(make_float2(__uint_as_float(oa[i]), __uint_as_float(oa[i + 1])),
                                          make_float2(__uint_as_float(os[i]), __uint_as_float(os[i + 1])), f);
                oa[i] = __float_as_uint(r2.x);
                oa[i + 1] = __float_as_uint(r2.y);
              }
            }
            tmem_st32(oacc_tmem + c * 32u, oa);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(Cfg::kBarORead));
          ++nfin;
        }
      }
    }
    if (ok && nt > 0)
      ok = mbar_wait(bar(Cfg::kBarOFull + (nt - 1) % Cfg::kSBufs), ((nt - 1) / Cfg::kSBufs) & 1, abort_flag,
                     args.err, kDevTimeoutMma);
    ok = __all_sync(0xffffffffu, ok) && nt > 0;
    if (ok && ws_mode) {
      // C5: this segment's partial (O unnormalised, m, mc, l) for the fold
      tc_fence_after();
      const bool store = m < n_rows;
      float* dst = args.part + ((((static_cast<size_t>(b) * args.Hq + g * kGroup + head) * args.L + r) * args.n_seg +
                                 seg_ws) * kPartFloats);
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
      // the last segment, folded with the ones before it (C5), then C4
      tc_fence_after();
      FoldScale f{1.0f, 1.0f};
      if (nfin == 0) acc = st;
      else f = fold_state(acc, st);
      const float inv_l = row_inv_l(acc);
      const bool store = m < n_rows;
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<__nv_bfloat16*>(args.o) +
          ((static_cast<size_t>(b) * args.Hq + g * kGroup + head) * args.L + r) * kHeadDim);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32], w[16];
        tmem_ld32_wait(o_tmem + c * 32u, o);
        if (nfin > 0) {
          uint32_t oa[32];
          tmem_ld32_wait(oacc_tmem + c * 32u, oa);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 r2 = fold_o2(make_float2(__uint_as_float(oa[i]), __uint_as_float(oa[i + 1])),
                                      make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f);
            o[i] = __float_as_uint(r2.x);
            o[i + 1] = __float_as_uint(r2.y);
          }
        }
        normalise32(o, inv_l, w);
        if (store) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[c * 4 + v4] = make_uint4(w[4 * v4 + 0], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        }
      }
    }
    if (C > 1) {                 // wide chunks run C = 1; kept so every thread meets the same barriers
      cluster_wait();
      if (pull_sync) cluster_sync();
    }
  } else if (warp == Cfg::kFoldWarp) {
    // --------------------------------------- fold and epilogue (narrow)
    // Per segment of this CTA: take its (m, l) from the softmax warp, wait
    // for its last P V, read O (the next segment's first P V may then clear
    // it) and finish the segment: the workspace partial, a fold in registers
    // (the cluster's first CTA) or a partial in shared memory (the others).
    // O is read through the 16x256b shape, so thread (m, u) holds row m's
    // columns 8r+2u, 8r+2u+1 as registers 4r, 4r+1 of each 64-column half.
    const int m = lane >> 2;                           // packed row 0..7
    const int u = lane & 3;
    const uint32_t o_tmem = tmem_base + Cfg::kOCol;    // lanes 0..31, reachable from warp 4
    const bool row_used = m < n_rows;
    const int head = row_used ? m / Lc : 0;
    const int r = row_used ? r0 + m % Lc : r0;
    const float2* stats = reinterpret_cast<const float2*>(smem + Cfg::kStatsOff);
    const float c = score_scale_log2();
    RowState acc = row_state_init();
    uint32_t acc0[32], acc1[32];                       // folded O (first CTA of the cluster)
    int nfin = 0;                                      // segments this CTA finished
    bool ok = run && no_error(args.err, abort_flag);
    const bool pushing = push && rank > 0;
    // the first CTA's partial slots and barrier, as addresses of the cluster
    const uint32_t lead_slots = pushing ? smem_addr_in_cta(sbase + Cfg::kPartOff, 0u) : 0u;
    const int my_first = seg_block_start(rank, ns, C);  // this CTA's first segment
    if (pushing) cluster_wait();                       // the first CTA's barriers are initialised

    auto finish_segment = [&](const RowState& sg, const uint32_t (&o0)[32], const uint32_t (&o1)[32]) {
      if (ws_mode) {
        if (row_used) {
          float* dst = args.part + ((((static_cast<size_t>(b) * args.Hq + g * kGroup + head) * args.L + r) *
                                     args.n_seg + seg_ws) * kPartFloats);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            *reinterpret_cast<float2*>(dst + 8 * q + 2 * u) =
                make_float2(__uint_as_float(o0[4 * q]), __uint_as_float(o0[4 * q + 1]));
            *reinterpret_cast<float2*>(dst + 64 + 8 * q + 2 * u) =
                make_float2(__uint_as_float(o1[4 * q]), __uint_as_float(o1[4 * q + 1]));
          }
          if (u == 0) *reinterpret_cast<float4*>(dst + 128) = make_float4(sg.m, sg.mc, sg.l, 0.0f);
        }
      } else if (rank == 0) {
        fold_segment_quad<false>(acc0, acc1, acc, acc, sg, sg, o0, o1, nfin == 0);
      } else if (pushing) {
        // into the first CTA's slot for this segment (push was chosen only
        // if every other CTA's segments fit there)
        if (row_used) {
          const uint32_t slot = lead_slots + static_cast<uint32_t>(my_first + nfin - s_first) * slot_bytes;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            st_cluster_f32x2(slot + 4u * static_cast<uint32_t>(m * 128 + 8 * q + 2 * u),
                             make_float2(__uint_as_float(o0[4 * q]), __uint_as_float(o0[4 * q + 1])));
            st_cluster_f32x2(slot + 4u * static_cast<uint32_t>(m * 128 + 64 + 8 * q + 2 * u),
                             make_float2(__uint_as_float(o1[4 * q]), __uint_as_float(o1[4 * q + 1])));
          }
          if (u == 0)
            st_cluster_f32x4(slot + 4u * static_cast<uint32_t>(n_rows * 128 + 4 * m),
                             make_float4(sg.m, sg.mc, sg.l, 0.0f));
        }
      } else if (static_cast<uint32_t>(nfin + 1) * slot_bytes > Cfg::kPartBytes) {
        // more segments than partial slots: the host sizes clusters so this
        // never happens; refuse rather than write past shared memory
        if (lane == 0) atomicCAS(args.err, 0u, static_cast<uint32_t>(kDevBadInput));
      } else if (row_used) {
        float* slot = reinterpret_cast<float*>(smem + Cfg::kPartOff + static_cast<uint32_t>(nfin) * slot_bytes);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          *reinterpret_cast<float2*>(slot + m * 128 + 8 * q + 2 * u) =
              make_float2(__uint_as_float(o0[4 * q]), __uint_as_float(o0[4 * q + 1]));
          *reinterpret_cast<float2*>(slot + m * 128 + 64 + 8 * q + 2 * u) =
              make_float2(__uint_as_float(o1[4 * q]), __uint_as_float(o1[4 * q + 1]));
        }
        if (u == 0) *reinterpret_cast<float4*>(slot + n_rows * 128 + 4 * m) = make_float4(sg.m, sg.mc, sg.l, 0.0f);
      }
      ++nfin;
    };

    int G = 0;
    for (int jb = 0; jb < nt && ok; jb += seg_len, ++G) {
      const int t_last = min(nt, jb + seg_len) - 1;           // local index of the segment's last tile
      // the stats are written after P(t_last), so P V(t_last - 3) is done and
      // the wait on P V(t_last) below is within one phase of its barrier
      ok = mbar_wait_idle(bar(Cfg::kBarStFull), G & 1, abort_flag, args.err, kDevTimeoutSoftmax, 128);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const float2 sv = stats[m];
      const RowState sg{sv.x, __fmul_rn(sv.x, c), sv.y};
      mbar_arrive(bar(Cfg::kBarStEmpty));
      ok = mbar_wait_idle(bar(Cfg::kBarOFull + t_last % Cfg::kSBufs), (t_last / Cfg::kSBufs) & 1, abort_flag,
                          args.err, kDevTimeoutMma, 32);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t o0[32], o1[32];
      tmem_ld_16x256b_x8_pair_wait(o_tmem, o_tmem + 64u, o0, o1);
      tc_fence_before();
      mbar_arrive(bar(Cfg::kBarORead));
      finish_segment(sg, o0, o1);
    }
    ok = ok && nt > 0;
    if (pushing) {
      // this CTA's partials are in the first CTA's shared memory (the
      // arrival releases the writes); it arrives whatever happened, so the
      // first CTA never waits for a CTA that gave up
      mbar_arrive_cluster(smem_addr_in_cta(bar(Cfg::kBarPart), 0u));
    } else if (C > 1) {
      cluster_wait();
      // partials in shared memory are complete: the cluster's first CTA reads
      // them after this barrier
      if (pull_sync) cluster_sync();
    }
    if (gather && rank > 0) {
      // this CTA's partials sit in its slots 0 .. n_mine-1; once the first
      // CTA has streamed its last tile, one bulk copy moves them into its
      // rings, at the place of their segments
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && mbar_wait_cluster(bar(Cfg::kBarGo), 0, abort_flag, args.err, kDevTimeoutSoftmax)) {
        const int n_mine = seg_block_start(rank + 1, ns, C) - my_first;
        bulk_copy_smem_to_cluster(
            smem_addr_in_cta(sbase + Cfg::kKOff + static_cast<uint32_t>(my_first - s_first) * slot_bytes, 0u),
            sbase + Cfg::kPartOff, static_cast<uint32_t>(n_mine) * slot_bytes, smem_addr_in_cta(bar(Cfg::kBarPart), 0u));
      }
      __syncwarp();
    }
    if (gather && rank == 0) {
      // every load of this CTA has landed and been consumed (its last P V is
      // done): the others may copy into its rings; signalled whatever
      // happened, so no CTA waits for one that gave up
      __syncwarp();
      if (lane == 0)
        for (int cr = 1; cr < C; ++cr) mbar_arrive_cluster(smem_addr_in_cta(bar(Cfg::kBarGo), static_cast<uint32_t>(cr)));
    }
    if ((push || gather) && rank == 0) {
      // this CTA's folded segments go to a slot of its own (push: after the
      // pushed ones; gather: its first partial slot, unused otherwise); warps
      // 0-3 fold once every fold warp writing to this CTA has arrived and
      // every copied byte has landed
      if (ok && row_used) {
        float* slot = reinterpret_cast<float*>(smem + Cfg::kPartOff +
                                               static_cast<uint32_t>(push ? ns - s_first : 0) * slot_bytes);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          *reinterpret_cast<float2*>(slot + m * 128 + 8 * q + 2 * u) =
              make_float2(__uint_as_float(acc0[4 * q]), __uint_as_float(acc0[4 * q + 1]));
          *reinterpret_cast<float2*>(slot + m * 128 + 64 + 8 * q + 2 * u) =
              make_float2(__uint_as_float(acc1[4 * q]), __uint_as_float(acc1[4 * q + 1]));
        }
        if (u == 0) *reinterpret_cast<float4*>(slot + n_rows * 128 + 4 * m) = make_float4(acc.m, acc.mc, acc.l, 0.0f);
      }
      mbar_arrive(bar(Cfg::kBarPart));                 // whatever happened, so warps 0-3 never wait for it
    }
    if (ok && !ws_mode && rank == 0 && !push && !gather) {
      // fold the other CTAs' segments, in segment order, from their shared
      // memory; the next segment's partial is loaded while this one folds
      int cr = 1;                                        // rank holding the segment being loaded
      auto load_seg = [&](int sgi, float4& sv, float2 (&ov)[16]) {
        while (cr + 1 < C && seg_block_start(cr + 1, ns, C) <= sgi) ++cr;
        const uint32_t k = static_cast<uint32_t>(sgi - seg_block_start(cr, ns, C));
        const uint32_t slot = smem_addr_in_cta(sbase + Cfg::kPartOff + k * slot_bytes, static_cast<uint32_t>(cr));
        if (row_used) {
          sv = ld_cluster_f32x4(slot + 4u * static_cast<uint32_t>(n_rows * 128 + 4 * m));
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            ov[q] = ld_cluster_f32x2(slot + 4u * static_cast<uint32_t>(m * 128 + 8 * q + 2 * u));
            ov[8 + q] = ld_cluster_f32x2(slot + 4u * static_cast<uint32_t>(m * 128 + 64 + 8 * q + 2 * u));
          }
        } else {
          sv = make_float4(-INFINITY, -INFINITY, 0.0f, 0.0f);
#pragma unroll
          for (int q = 0; q < 16; ++q) ov[q] = make_float2(0.0f, 0.0f);
        }
      };
      // the same arithmetic as fold_segment_quad on row A: fold_state, then
      // fold_o2 on each pair of the thread's 32 columns
      auto fold_seg = [&](const float4& sv, const float2 (&ov)[16]) {
        const FoldScale f = fold_state(acc, RowState{sv.x, sv.y, sv.z});
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float2 r0 = fold_o2(make_float2(__uint_as_float(acc0[4 * q]), __uint_as_float(acc0[4 * q + 1])), ov[q], f);
          const float2 r1 =
              fold_o2(make_float2(__uint_as_float(acc1[4 * q]), __uint_as_float(acc1[4 * q + 1])), ov[8 + q], f);
          acc0[4 * q] = __float_as_uint(r0.x);
          acc0[4 * q + 1] = __float_as_uint(r0.y);
          acc1[4 * q] = __float_as_uint(r1.x);
          acc1[4 * q + 1] = __float_as_uint(r1.y);
        }
      };
      float4 svA, svB;
      float2 ovA[16], ovB[16];
      int sgi = s_first;                                 // the first segment another CTA ran
      const bool pull = pull_sync;
      if (pull && sgi < ns) load_seg(sgi, svA, ovA);
#pragma unroll 1
      while (pull && sgi < ns) {
        if (sgi + 1 < ns) load_seg(sgi + 1, svB, ovB);
        fold_seg(svA, ovA);
        if (++sgi >= ns) break;
        if (sgi + 1 < ns) load_seg(sgi + 1, svA, ovA);
        fold_seg(svB, ovB);
        ++sgi;
      }
      // C4 into the rows' outputs: thread (m, u) stores its 32 columns
      const float inv_l = row_inv_l(acc);
      if (row_used) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(
            static_cast<__nv_bfloat16*>(args.o) +
            ((static_cast<size_t>(b) * args.Hq + g * kGroup + head) * args.L + r) * kHeadDim);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          dst[(8 * q + 2 * u) >> 1] = pack_bf16x2(__fmul_rn(__uint_as_float(acc0[4 * q]), inv_l),
                                                  __fmul_rn(__uint_as_float(acc0[4 * q + 1]), inv_l));
          dst[(64 + 8 * q + 2 * u) >> 1] = pack_bf16x2(__fmul_rn(__uint_as_float(acc1[4 * q]), inv_l),
                                                       __fmul_rn(__uint_as_float(acc1[4 * q + 1]), inv_l));
        }
      }
    }
  } else {
    // ------------------------------------- softmax, four threads per row (narrow)
    // Rows 0..7 live in TMEM lanes 0..7; the 16x256b load gives each quad of
    // lanes 4i..4i+3 row i (and lanes 8..15, which alias rows 0..7), thread
    // u holding keys 8r+2u, 8r+2u+1 (r = 0..15), so the row's 128
    // exponentials are spread over four threads.
    const int m = lane >> 2;                           // packed row 0..7
    const int u = lane & 3;
    const uint32_t o_tmem = tmem_base + Cfg::kOCol;    // warp 0: lanes 0..31
    const bool row_used = m < n_rows;
    const int r = row_used ? r0 + m % Lc : r0;         // unused rows take the sub-chunk's first position
    const int pos = pos0 + r;
    float2* stats = reinterpret_cast<float2*>(smem + Cfg::kStatsOff);
    RowState st = row_state_init();
    int js = 0;                                        // tile index within its segment (j0 starts one)
    int G = 0;                                         // segments handed to the fold warp
    bool ok = run && no_error(args.err, abort_flag);
    for (int j = 0; j < nt && ok; ++j) {                    // j: tile j0 + j
      ok = mbar_wait_hint(bar(Cfg::kBarSFull + j % Cfg::kSBufs), (j / Cfg::kSBufs) & 1, abort_flag, args.err,
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
      const int jt = j0 + j;
      const bool seg_start = (js == 0);
      if (++js == seg_len) js = 0;
      const bool seg_end = (js == 0) || (j == nt - 1);
      if (seg_start) st = row_state_init();
      uint32_t p[16];
      const float alpha = (jt == n_kv - 1) ? row_softmax_tile_quad<true>(x, u, pos - jt * kTileKeys + 1, st, p)
                                           : row_softmax_tile_quad<false>(x, u, kTileKeys, st, p);
      if (!seg_start && __any_sync(0xffffffffu, alpha != 1.0f)) {
        // rescale O (rows in lanes 0..31 through the 32x32b shape; lane L takes
        // the factor of row L % 8, rows 8..31 are never stored)
        ok = mbar_wait(bar(Cfg::kBarOFull + (j - 1) % Cfg::kSBufs), ((j - 1) / Cfg::kSBufs) & 1, abort_flag,
                       args.err, kDevTimeoutMma);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float a_lane = __shfl_sync(0xffffffffu, alpha, 4 * (lane & 7));
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32_wait(o_tmem + cc * 32u, o);
          rescale32(o, a_lane);
          tmem_st32(o_tmem + cc * 32u, o);
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
      if (seg_end) {
        // C5: hand the finished segment's (m, l) to the fold warp, once it has
        // read the previous segment's
        if (G > 0) {
          ok = mbar_wait(bar(Cfg::kBarStEmpty), (G - 1) & 1, abort_flag, args.err, kDevTimeoutSoftmax);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        if (u == 0) stats[m] = make_float2(st.m, st.l);
        mbar_arrive(bar(Cfg::kBarStFull));
        ++G;
      }
    }
    if (C > 1) {
      cluster_wait();
      if (pull_sync) cluster_sync();
    }
  }

  if ((push || gather) && rank == 0 && warp < 4) {
    // ---------------------- final fold of a push or gather cluster (narrow)
    // Slots 0 .. ns-s_first-1 (push: the partial slots; gather: the K/V
    // rings) hold segments s_first .. ns-1; this CTA's folded segments 0 ..
    // s_first-1 are in the partial slot after them (push) or in the first
    // partial slot (gather).  Thread t folds packed
    // row t/16, columns 8(t%16) .. +7, left to right (C5), then C4; the
    // operations and their order are those of the fold warp's serial fold.
    const int r = threadIdx.x >> 4;
    const int cb = threadIdx.x & 15;
    bool ok = mbar_wait_cluster(bar(Cfg::kBarPart), 0, abort_flag, args.err, kDevTimeoutSoftmax);
    ok = ok && (*abort_flag == 0);
    if (ok && r < n_rows) {
      const float* slots = reinterpret_cast<const float*>(smem + (push ? Cfg::kPartOff : Cfg::kKOff));
      const float* own = reinterpret_cast<const float*>(smem + Cfg::kPartOff);
      const uint32_t slot_floats = slot_bytes / 4u;
      const int n_push = ns - s_first;
      auto load = [&](int k, float4& st, float4& oa, float4& ob) {
        const float* sl = (k == n_push) ? (push ? slots + static_cast<uint32_t>(k) * slot_floats : own)
                                        : slots + static_cast<uint32_t>(k) * slot_floats;
        st = *reinterpret_cast<const float4*>(sl + n_rows * 128 + 4 * r);
        oa = *reinterpret_cast<const float4*>(sl + r * 128 + 8 * cb);
        ob = *reinterpret_cast<const float4*>(sl + r * 128 + 8 * cb + 4);
      };
      float4 st, oa, ob;
      load(n_push, st, oa, ob);
      RowState acc{st.x, st.y, st.z};
      float o[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
      float4 nst, noa, nob;
      if (n_push > 0) load(0, nst, noa, nob);
#pragma unroll 1
      for (int k = 0; k < n_push; ++k) {
        const float4 cst = nst, coa = noa, cob = nob;
        if (k + 1 < n_push) load(k + 1, nst, noa, nob);           // next slot in flight while this one folds
        const FoldScale f = fold_state(acc, RowState{cst.x, cst.y, cst.z});
        const float os[8] = {coa.x, coa.y, coa.z, coa.w, cob.x, cob.y, cob.z, cob.w};
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 r2 = fold_o2(make_float2(o[i], o[i + 1]), make_float2(os[i], os[i + 1]), f);
          o[i] = r2.x;
          o[i + 1] = r2.y;
        }
      }
      const float inv_l = row_inv_l(acc);
      const int head = r / Lc;
      const int rr = r0 + r % Lc;
      uint4 packed;
      packed.x = pack_bf16x2(__fmul_rn(o[0], inv_l), __fmul_rn(o[1], inv_l));
      packed.y = pack_bf16x2(__fmul_rn(o[2], inv_l), __fmul_rn(o[3], inv_l));
      packed.z = pack_bf16x2(__fmul_rn(o[4], inv_l), __fmul_rn(o[5], inv_l));
      packed.w = pack_bf16x2(__fmul_rn(o[6], inv_l), __fmul_rn(o[7], inv_l));
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) +
                                ((static_cast<size_t>(b) * args.Hq + g * kGroup + head) * args.L + rr) * kHeadDim +
                                8 * cb) = packed;
    }
  }

  // the first CTA has read every partial: the others may leave
  if (C > 1) cluster_sync();
  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::kQkWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <bool kWide, int kNumSBufs>
static cudaError_t launch_packed_t(const CUtensorMap& tk, const CUtensorMap& tv, const PackedArgs& a, int n_sub,
                                   cudaStream_t s) {
  using Cfg = PackedCfg<kWide, kNumSBufs>;
  static_assert(Cfg::kSmemBytes <= 227u * 1024u, "shared memory budget");
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kb_decode_kernel<kWide, kNumSBufs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const bool ws_mode = a.part != nullptr;
  const int C = ws_mode ? 1 : a.cluster;
  const unsigned grid = static_cast<unsigned>((ws_mode ? a.n_seg : C) * n_sub * a.B * a.Hkv);
  if (C <= 1) {
    kb_decode_kernel<kWide, kNumSBufs><<<grid, Cfg::kThreads, Cfg::kSmemBytes, s>>>(tk, tv, a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kb_decode_kernel<kWide, kNumSBufs>, tk, tv, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_packed(const CUtensorMap& tk, const CUtensorMap& tv, const PackedArgs& a, int n_sub,
                          cudaStream_t s) {
  // narrow when at most 8 rows are packed (two query rows per head); wide
  // chunks fold their segments in TMEM (two S buffers) unless the partials
  // go to a workspace
  if (a.L <= 2) return launch_packed_t<false, 3>(tk, tv, a, n_sub, s);
  if (a.part != nullptr) return launch_packed_t<true, 3>(tk, tv, a, n_sub, s);
  return launch_packed_t<true, 2>(tk, tv, a, n_sub, s);
}

// How many clusters of 2, 4 and 8 CTAs of the narrow packed kernel the
// current device runs at once (0 when it runs none): a cluster needs that
// many SMs of one GPC free together, so large clusters fit fewer times than
// the SM count suggests.
void packed_cluster_capacity(int (&active)[4]) {
  using Cfg = PackedCfg<false, 3>;
  for (int i = 0; i < 4; ++i) active[i] = 0;
  if (cudaFuncSetAttribute(kb_decode_kernel<false, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(Cfg::kSmemBytes)) != cudaSuccess) {
    (void)cudaGetLastError();
    return;
  }
  for (int i = 1, c = 2; i < 4; ++i, c *= 2) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(c), 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kb_decode_kernel<false, 3>, &cfg) == cudaSuccess) active[i] = n;
    else (void)cudaGetLastError();
  }
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
