// kb_decode.cu -- one-token decode over a contiguous KV cache (KernelBraid
// README, "Usage": unified_decode over the same KV context, whose output must
// equal the prefill row bit for bit; "Features": one query token per decode
// call).
//
// One CTA per (batch, KV head).  The four query heads of the GQA group are
// packed into rows 0..3 of the M=128 MMA (rows 4..7 are zero and row groups
// 8..127 alias rows 0..7 through a zero stride-byte-offset descriptor), so
// decode issues the very same tcgen05.mma shape, k-order and row softmax as
// prefill and every packed row reproduces the prefill row exactly.  K/V tiles
// stream through a three-deep TMA ring; S is double-buffered in TMEM so the
// next Q K^T overlaps the current softmax.
//   warp 0  softmax (TMEM lanes 0..31; lanes 0..3 are the four heads)
//   warp 1  TMA producer (one lane)
//   warp 2  TMEM allocator + MMA issuer (one lane)
#include "kb_contract.cuh"
#include "kb_launch.h"

namespace kb {

struct DecodeCfg {
  static constexpr int kThreads = 96;
  static constexpr int kStages = 3;
  static constexpr uint32_t kTmemCols = 512;   // S0, S1, O (128 columns each)
  static constexpr uint32_t kQAtom = 1024;     // 8 rows x 128 bytes, one per d-slab
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = 2 * kQAtom;
  static constexpr uint32_t kVOff = kKOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kBarKFull = 0;
  static constexpr int kBarKEmpty = kBarKFull + kStages;
  static constexpr int kBarVFull = kBarKEmpty + kStages;
  static constexpr int kBarVEmpty = kBarVFull + kStages;
  static constexpr int kBarSFull = kBarVEmpty + kStages;   // 2 (double-buffered S)
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarOFull = kBarPFull + 1;
  static constexpr int kBarDrain = kBarOFull + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemUsed = kMiscOff + 16;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
};

__device__ __forceinline__ void decode_drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 50000000ull) break;
}

__global__ void __launch_bounds__(DecodeCfg::kThreads, 1)
kb_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const DecodeArgs args) {
  using Cfg = DecodeCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) { return smem_addr(bars + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x / args.Hkv;
  const int g = blockIdx.x % args.Hkv;
  const int ctx = args.ctx;
  const int n_kv = (ctx - 1) / kTileKeys + 1;     // C1: KV tiles 0..floor((ctx-1)/128)

  // Q rows 0..3 = heads 4g..4g+3, rows 4..7 = 0, written in the 128-byte
  // swizzled layout the MMA descriptor expects (16-byte chunk c of row r
  // sits at chunk c ^ r).
  {
    const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.q) +
                                                       (static_cast<size_t>(b) * args.Hq + g * kGroup) * kHeadDim);
    for (int idx = threadIdx.x; idx < 8 * 16; idx += Cfg::kThreads) {
      const int row = idx >> 4;
      const int c = idx & 15;
      const int slab = c >> 3;
      const int cc = c & 7;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (row < kGroup) val = __ldg(qsrc + row * (kHeadDim / 8) + c);
      *reinterpret_cast<uint4*>(smem + Cfg::kQOff + slab * Cfg::kQAtom + row * 128 + ((cc ^ row) << 4)) = val;
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i) mbar_init(bar(i), i == Cfg::kBarPFull ? 32u : 1u);
    misc[1] = (*reinterpret_cast<volatile uint32_t*>(args.err) != 0) ? 1u : 0u;
    fence_mbar_init();
  }
  fence_proxy_async_smem();   // generic-proxy Q writes -> visible to the tensor core
  if (warp == 2) {
    tmem_alloc(sbase + Cfg::kMiscOff, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const bool skip = (*abort_flag != 0);

  if (warp == 1) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !skip) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      const uint64_t stream_once = l2_policy_evict_first();
      const int z = b * args.Hkv + g;
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int slot = j % Cfg::kStages;
        const uint32_t use = j / Cfg::kStages;
        if (j >= Cfg::kStages)
          ok = mbar_wait(bar(Cfg::kBarKEmpty + slot), (use - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        if (!ok) break;
        const uint32_t kdst = sbase + Cfg::kKOff + slot * kTileBytes;
        mbar_arrive_expect_tx(bar(Cfg::kBarKFull + slot), kTileBytes);
        tma_load_3d_hint(kdst, &tmap_k, 0, j * kTileKeys, z, bar(Cfg::kBarKFull + slot), stream_once);
        tma_load_3d_hint(kdst + kSlabBytes, &tmap_k, 64, j * kTileKeys, z, bar(Cfg::kBarKFull + slot), stream_once);
        if (j >= Cfg::kStages)
          ok = mbar_wait(bar(Cfg::kBarVEmpty + slot), (use - 1) & 1, abort_flag, args.err, kDevTimeoutSlot);
        if (!ok) { issued = 2 * j + 1; break; }
        const uint32_t vdst = sbase + Cfg::kVOff + slot * kTileBytes;
        mbar_arrive_expect_tx(bar(Cfg::kBarVFull + slot), kTileBytes);
        tma_load_3d_hint(vdst, &tmap_v, 0, j * kTileKeys, z, bar(Cfg::kBarVFull + slot), stream_once);
        tma_load_3d_hint(vdst + kSlabBytes, &tmap_v, 64, j * kTileKeys, z, bar(Cfg::kBarVFull + slot), stream_once);
        issued = 2 * j + 2;
      }
      if (!ok) {
        for (int x = (issued > 2 * Cfg::kStages ? issued - 2 * Cfg::kStages : 0); x < issued; ++x) {
          const int j = x >> 1;
          decode_drain_wait(bar(((x & 1) ? Cfg::kBarVFull : Cfg::kBarKFull) + j % Cfg::kStages),
                            (j / Cfg::kStages) & 1);
        }
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && !skip) {
      const uint32_t q_saddr = sbase + Cfg::kQOff;
      bool ok = mbar_wait(bar(Cfg::kBarKFull), 0, abort_flag, args.err, kDevTimeoutTma);
      if (ok) {
        tc_fence_after();
        issue_qk(tmem_base, q_saddr, 0u, Cfg::kQAtom, sbase + Cfg::kKOff);
        tc_commit(bar(Cfg::kBarSFull));
        tc_commit(bar(Cfg::kBarKEmpty));
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j + 1 < n_kv) {
          const int jn = j + 1;
          const int slot = jn % Cfg::kStages;
          ok = mbar_wait(bar(Cfg::kBarKFull + slot), (jn / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
          // S buffer jn%2 held P of tile j-1: free once that P V has finished
          if (ok && jn >= 2) ok = mbar_wait(bar(Cfg::kBarOFull), (j - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          issue_qk(tmem_base + (jn & 1) * 128u, q_saddr, 0u, Cfg::kQAtom, sbase + Cfg::kKOff + slot * kTileBytes);
          tc_commit(bar(Cfg::kBarSFull + (jn & 1)));
          tc_commit(bar(Cfg::kBarKEmpty + slot));
        }
        const int slot = j % Cfg::kStages;
        ok = mbar_wait(bar(Cfg::kBarPFull), j & 1, abort_flag, args.err, kDevTimeoutSoftmax);
        if (ok) ok = mbar_wait(bar(Cfg::kBarVFull + slot), (j / Cfg::kStages) & 1, abort_flag, args.err, kDevTimeoutTma);
        if (!ok) break;
        tc_fence_after();
        issue_pv(tmem_base + 256u, tmem_base + (j & 1) * 128u, sbase + Cfg::kVOff + slot * kTileBytes, j == 0);
        tc_commit(bar(Cfg::kBarOFull));
        tc_commit(bar(Cfg::kBarVEmpty + slot));
      }
      if (!ok) {
        tc_commit(bar(Cfg::kBarDrain));
        decode_drain_wait(bar(Cfg::kBarDrain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    const uint32_t o_tmem = tmem_base + 256u;   // warp 0: lanes 0..31, lane offset 0
    RowState st = row_state_init();
    bool ok = !skip;
    for (int j = 0; j < n_kv && ok; ++j) {
      ok = mbar_wait(bar(Cfg::kBarSFull + (j & 1)), (j >> 1) & 1, abort_flag, args.err, kDevTimeoutMma);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tmem = tmem_base + (j & 1) * 128u;
      uint32_t s[128];
      tmem_ld128_wait(s_tmem, s);
      uint32_t p[64];
      const float alpha = (j == n_kv - 1) ? row_softmax_tile<true>(s, ctx - j * kTileKeys, st, p)
                                          : row_softmax_tile<false>(s, kTileKeys, st, p);
      if (j > 0) {
        ok = mbar_wait(bar(Cfg::kBarOFull), (j - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
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
      mbar_arrive(bar(Cfg::kBarPFull));
    }
    if (ok) ok = mbar_wait(bar(Cfg::kBarOFull), (n_kv - 1) & 1, abort_flag, args.err, kDevTimeoutMma);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const float inv_l = row_inv_l(st);
      const bool store = lane < kGroup;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o) +
                                            (static_cast<size_t>(b) * args.Hq + g * kGroup + (store ? lane : 0)) *
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
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t s) {
  static_assert(DecodeCfg::kSmemUsed <= 227u * 1024u, "shared memory budget");
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kb_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(DecodeCfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  kb_decode_kernel<<<static_cast<unsigned>(a.B * a.Hkv), DecodeCfg::kThreads, DecodeCfg::kSmemBytes, s>>>(tk, tv, a);
  return cudaGetLastError();
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
