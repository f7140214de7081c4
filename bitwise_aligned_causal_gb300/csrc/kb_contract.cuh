// kb_contract.cuh -- the numerical contract shared by every entry point.
//
// The KernelBraid README ("Method") requires one numerical contract that
// connects full-sequence prefill, partitioned (chunked) forward and
// one-token decode, so that the three produce bitwise-identical output rows
// for the same inputs and context ("Advantages"; the "Usage" example compares
// the raw bf16 bits).  The pages do not print the contract's contents, so it
// is fixed here, version 3:
//
//  C1 One KV tile of 128 keys, anchored at key 0, visited in ascending order
//     0..floor(p/128) for a row at absolute position p.  Prefill/chunk query
//     tiles are aligned to absolute multiples of 128, so every row of a tile
//     ends on the same KV tile and no row ever visits a fully masked tile.
//  C2 One MMA: tcgen05.mma.cta_group::1.kind::f16, bf16 x bf16 -> fp32,
//     M=128 N=128 K=16.  S = Q K^T and O += P V each issue eight of them in
//     ascending K order; S is A/B from shared memory, P V reads P from TMEM.
//  C3 One thread owns one row of S and O (TMEM lane = row).  All row math is
//     the functions below; data-dependent choices (when the reference max
//     moves, which keys are masked) are per row only.
//  C4 One normalisation: o = bf16_rn(O * rcp_rn(l)).
//  C5 A fixed, length-determined split of the KV range: a row's key tiles
//     are cut into segments of kSegTiles tiles anchored at tile 0; each
//     segment runs C1-C3 from the fresh state (its first P V clears the
//     accumulator) and the segments are folded left to right by fold_state /
//     fold_o below, then C4.  A row whose keys fit in one segment gets the
//     plain online-softmax bits.  The segment length is the same for every
//     entry point, so a decode may give each segment its own CTA while
//     prefill folds the same segments in order.  (The *_seg entry points take
//     other segment lengths; a length of at least the row's tile count is
//     the unsplit online softmax, version 2's default.)
//
// Every floating-point operation below is an explicit round-to-nearest
// intrinsic, so the compiler cannot contract or reorder them differently in
// different kernels.
#pragma once

#include <cstdint>
#include "kb_ptx.cuh"

namespace kb {

constexpr int kHeadDim = 128;      // D
constexpr int kTileKeys = 128;     // keys per KV tile (C1)
constexpr int kTileRows = 128;     // query rows per tile = MMA M (C2)
constexpr int kGroup = 4;          // query heads per KV head (32 / 8)
constexpr int kContractVersion = 3;
constexpr int kSegTiles = 8;       // C5: keys per segment = 8 * 128 = 1024

// c = log2(e) / sqrt(128) = 0.1275174308245986852... rounded to the nearest
// fp32, bit pattern 0x3E0293EE.  The softmax weight of score s against the
// running max m is 2^(s*c - m*c) = e^((s - m) / sqrt(128)).
constexpr uint32_t kScoreScaleLog2Bits = 0x3E0293EEu;
__device__ __forceinline__ float score_scale_log2() { return __uint_as_float(kScoreScaleLog2Bits); }

constexpr uint32_t kTileBytes = kTileRows * kHeadDim * 2;   // one bf16 128x128 tile
constexpr uint32_t kSlabBytes = kTileBytes / 2;             // one 128 x 64 swizzled slab

// Instruction descriptors for the two products (C2).
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0);  // B = K tile, K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 1);  // B = V tile, MN-major

// Descriptor of k-step kk (0..7) of a K-major 128-row tile stored as two
// 128-byte-swizzled slabs (d 0..63, d 64..127).  `sbo` is the distance
// between 8-row groups: 1024 for a full tile, 0 when all row groups alias one
// 8-row atom (decode, where only rows 0..3 carry queries).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_saddr, int kk, uint32_t sbo, uint32_t slab_bytes) {
  const uint32_t a = tile_saddr + static_cast<uint32_t>(kk >> 2) * slab_bytes + static_cast<uint32_t>(kk & 3) * 32u;
  return smem_desc_sw128(a, 16u, sbo);
}

// Descriptor of k-step kk (keys 16kk..16kk+15) of a V tile: keys are rows,
// d is contiguous (MN-major), slabs of 64 d-columns 16 KB apart.
__device__ __forceinline__ uint64_t desc_v(uint32_t tile_saddr, int kk) {
  return smem_desc_sw128(tile_saddr + static_cast<uint32_t>(kk) * 2048u, kSlabBytes, 1024u);
}

// Issue S = Q K^T for one query tile (C2: eight K=16 steps, ascending).
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint32_t q_saddr, uint32_t q_sbo, uint32_t q_slab,
                                         uint32_t k_saddr) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ss(s_tmem, desc_kmajor(q_saddr, kk, q_sbo, q_slab), desc_kmajor(k_saddr, kk, 1024u, kSlabBytes), kIdescQK,
           kk > 0 ? 1u : 0u);
}

// Issue O (+)= P V (C2).  P sits in TMEM as bf16 pairs, 8 columns per K step.
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_saddr, bool first_tile) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(o_tmem, p_tmem + static_cast<uint32_t>(kk) * 8u, desc_v(v_saddr, kk), kIdescPV,
           (first_tile && kk == 0) ? 0u : 1u);
}

// Per-row running state of the online softmax.
struct RowState {
  float m;   // reference max of the raw scores q.k (unscaled); -inf before the first tile
  float mc;  // m * c, rounded to fp32
  float l;   // running sum of the fp32 weights
};

__device__ __forceinline__ RowState row_state_init() { return RowState{-INFINITY, -INFINITY, 0.0f}; }

// The reference max moves only when a tile's max exceeds it by more than
// this many raw score units (64 * c = 8.16 in log2 units), so weights stay
// below 2^8.2 and the O rescale is rare.  The decision is per row.
constexpr float kRescaleThresholdRaw = 64.0f;

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// One KV tile of the online softmax for one row (C3).
//
//  s[k]     raw scores q.k of keys 128j+k (fp32 bit patterns from TMEM)
//  kMasked  true only on the row's last tile; then keys k >= n_valid are
//           masked to -inf (a select, so an all-visible tile gives the same
//           bits either way)
//  p        out: the weights rounded to bf16, packed two per word, key 2i in
//           the low half of p[i]
//  returns  alpha, the factor the row's O accumulator must be scaled by
//           before this tile's P V is added (exactly 1.0 when the reference
//           max did not move, exactly 0.0 on the first tile)
//
//  t     = max_k s[k]                                          (exact)
//  if t - m > 64 (always on the first tile, where m = -inf):
//        m' = t, mc' = m' * c, alpha = 2^(fma(m, c, -mc'))
//  else  m' = m, mc' = mc, alpha = 1
//  w[k]  = 2^(fma(s[k], c, -mc'))   (masked keys -> +0)
//  l'    = fma(l, alpha, sum_k w[k]), the sum taken as eight strided partial
//          sums (k mod 8, ascending k) combined as ((0+1)+(2+3))+((4+5)+(6+7))
// with c = log2(e)/sqrt(128) in fp32 and 2^x the hardware ex2.approx.ftz.
template <bool kMasked>
__device__ __forceinline__ float row_softmax_tile(const uint32_t (&s)[128], int n_valid, RowState& st,
                                                  uint32_t (&p)[64]) {
  const float c = score_scale_log2();
  float x[128];
#pragma unroll
  for (int k = 0; k < 128; ++k) {
    x[k] = __uint_as_float(s[k]);
    if (kMasked) x[k] = (k < n_valid) ? x[k] : -INFINITY;
  }

  // exact row max (max is order-free): 128 values in 64 three- and two-input
  // maxima, five levels deep
  float m1[44];
#pragma unroll
  for (int i = 0; i < 42; ++i) m1[i] = max3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  m1[42] = x[126];
  m1[43] = x[127];
  float m2[16];
#pragma unroll
  for (int i = 0; i < 14; ++i) m2[i] = max3(m1[3 * i], m1[3 * i + 1], m1[3 * i + 2]);
  m2[14] = m1[42];
  m2[15] = m1[43];
  float m3[6];
#pragma unroll
  for (int i = 0; i < 5; ++i) m3[i] = max3(m2[3 * i], m2[3 * i + 1], m2[3 * i + 2]);
  m3[5] = m2[15];
  const float tile_max = fmaxf(max3(m3[0], m3[1], m3[2]), max3(m3[3], m3[4], m3[5]));

  float alpha = 1.0f;
  if (__fsub_rn(tile_max, st.m) > kRescaleThresholdRaw) {
    const float mc_new = __fmul_rn(tile_max, c);
    alpha = ex2_approx(__fmaf_rn(st.m, c, -mc_new));
    st.m = tile_max;
    st.mc = mc_new;
  }
  const float2 c2 = make_float2(c, c);
  const float2 nmc2 = make_float2(-st.mc, -st.mc);

  float2 acc[4];
#pragma unroll
  for (int k = 0; k < 128; k += 2) {
    const float2 arg = __ffma2_rn(make_float2(x[k], x[k + 1]), c2, nmc2);
    const float w0 = ex2_approx(arg.x);
    const float w1 = ex2_approx(arg.y);
    x[k] = w0;
    x[k + 1] = w1;
    const int a = (k & 7) >> 1;
    if (k < 8) acc[a] = make_float2(w0, w1);
    else acc[a] = __fadd2_rn(acc[a], make_float2(w0, w1));
  }
  const float tile_sum = __fadd_rn(__fadd_rn(__fadd_rn(acc[0].x, acc[0].y), __fadd_rn(acc[1].x, acc[1].y)),
                                   __fadd_rn(__fadd_rn(acc[2].x, acc[2].y), __fadd_rn(acc[3].x, acc[3].y)));
#pragma unroll
  for (int i = 0; i < 64; ++i) p[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);

  st.l = __fmaf_rn(st.l, alpha, tile_sum);
  return alpha;
}

// The same tile step with a row spread over four threads (a quad of lanes
// 4i..4i+3, thread u = lane % 4), as the 16x256b TMEM load lays it out:
// thread u holds keys 8r+2u and 8r+2u+1 (x[2r], x[2r+1]) for r = 0..15, which
// are exactly the keys of the partial sums k mod 8 = 2u and 2u+1 above.  The
// max and the pair sums are combined across the quad with shuffles in the
// same order as the single-thread tree, so the bits are the same; p[r] is the
// bf16 pair of keys 8r+2u, 8r+2u+1 (TMEM column 4r+u of P).  All 32 lanes of
// the warp must call it together.
template <bool kMasked>
__device__ __forceinline__ float row_softmax_tile_quad(float (&x)[32], int u, int n_valid, RowState& st,
                                                       uint32_t (&p)[16]) {
  const float c = score_scale_log2();
  if (kMasked) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      x[2 * r] = (8 * r + 2 * u < n_valid) ? x[2 * r] : -INFINITY;
      x[2 * r + 1] = (8 * r + 2 * u + 1 < n_valid) ? x[2 * r + 1] : -INFINITY;
    }
  }
  // exact maximum (order-free): 32 values in 16 three- and two-input maxima
  float mx[12];
#pragma unroll
  for (int i = 0; i < 10; ++i) mx[i] = max3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  mx[10] = x[30];
  mx[11] = x[31];
  float my[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) my[i] = max3(mx[3 * i], mx[3 * i + 1], mx[3 * i + 2]);
  float tile_max = fmaxf(max3(my[0], my[1], my[2]), my[3]);
  tile_max = fmaxf(tile_max, __shfl_xor_sync(0xffffffffu, tile_max, 1));
  tile_max = fmaxf(tile_max, __shfl_xor_sync(0xffffffffu, tile_max, 2));

  float alpha = 1.0f;
  if (__fsub_rn(tile_max, st.m) > kRescaleThresholdRaw) {
    const float mc_new = __fmul_rn(tile_max, c);
    alpha = ex2_approx(__fmaf_rn(st.m, c, -mc_new));
    st.m = tile_max;
    st.mc = mc_new;
  }
  const float2 c2 = make_float2(c, c);
  const float2 nmc2 = make_float2(-st.mc, -st.mc);
  float2 acc;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float2 arg = __ffma2_rn(make_float2(x[2 * r], x[2 * r + 1]), c2, nmc2);
    const float w0 = ex2_approx(arg.x);
    const float w1 = ex2_approx(arg.y);
    acc = (r == 0) ? make_float2(w0, w1) : __fadd2_rn(acc, make_float2(w0, w1));
    p[r] = pack_bf16x2(w0, w1);
  }
  const float s_pair = __fadd_rn(acc.x, acc.y);                                      // acc[u].x + acc[u].y
  const float s_half = __fadd_rn(s_pair, __shfl_xor_sync(0xffffffffu, s_pair, 1)); // (0+1) or (2+3)
  const float tile_sum = __fadd_rn(s_half, __shfl_xor_sync(0xffffffffu, s_half, 2));
  st.l = __fmaf_rn(st.l, alpha, tile_sum);
  return alpha;
}

// Scale 32 accumulator columns by alpha (bit-neutral when alpha == 1).
__device__ __forceinline__ void rescale32(uint32_t (&o)[32], float alpha) {
  const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 r = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
    o[i] = __float_as_uint(r.x);
    o[i + 1] = __float_as_uint(r.y);
  }
}

// C4: final normalisation of 32 accumulator columns into 16 bf16 pairs.
__device__ __forceinline__ void normalise32(const uint32_t (&o)[32], float inv_l, uint32_t (&out)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    out[i] = pack_bf16x2(__fmul_rn(__uint_as_float(o[2 * i]), inv_l), __fmul_rn(__uint_as_float(o[2 * i + 1]), inv_l));
}

__device__ __forceinline__ float row_inv_l(const RowState& st) { return __frcp_rn(st.l); }

// C5 fold of a segment's (m, mc, l, O) into the accumulated (m, mc, l, O) of
// the segments before it: both are brought to the larger reference max M,
// the side already at M by exactly 1, the other by 2^(m c - M c):
//   l <- fma(l_acc, a, l_seg * b),   O <- fma(O_acc, a, O_seg * b).
// The first segment is taken as it is (no fold).
struct FoldScale {
  float a;  // factor of the accumulated segments
  float b;  // factor of the new segment
};

__device__ __forceinline__ FoldScale fold_state(RowState& acc, const RowState& seg) {
  const float c = score_scale_log2();
  const bool keep = acc.m >= seg.m;
  const float mc = keep ? acc.mc : seg.mc;                 // M * c, as computed when M was set
  const float a = keep ? 1.0f : ex2_approx(__fmaf_rn(acc.m, c, -mc));
  const float b = (seg.m >= acc.m) ? 1.0f : ex2_approx(__fmaf_rn(seg.m, c, -mc));
  acc.l = __fmaf_rn(acc.l, a, __fmul_rn(seg.l, b));
  acc.m = keep ? acc.m : seg.m;
  acc.mc = mc;
  return FoldScale{a, b};
}

__device__ __forceinline__ float fold_o(float o_acc, float o_seg, FoldScale f) {
  return __fmaf_rn(o_acc, f.a, __fmul_rn(o_seg, f.b));
}

// fold_o on two columns at once, as packed f32x2 operations (the same two
// round-to-nearest operations per column, so the same bits).
__device__ __forceinline__ float2 fold_o2(float2 o_acc, float2 o_seg, FoldScale f) {
  return __ffma2_rn(o_acc, make_float2(f.a, f.a), __fmul2_rn(o_seg, make_float2(f.b, f.b)));
}

// C5 fold of one finished segment into a thread's share of the folded O, in
// the register layout of two 16x256b.x8 TMEM loads (columns 0-63 and
// 64-127): registers 4r, 4r+1 of each half belong to the thread's row A,
// 4r+2, 4r+3 to its row B.  `first` takes the segment as it is.  kRowB false:
// only row A is real (the B registers are ignored).
template <bool kRowB>
__device__ __forceinline__ void fold_segment_quad(uint32_t (&acc0)[32], uint32_t (&acc1)[32], RowState& accA,
                                                  RowState& accB, const RowState& segA, const RowState& segB,
                                                  const uint32_t (&o0)[32], const uint32_t (&o1)[32], bool first) {
  if (first) {
    accA = segA;
    if (kRowB) accB = segB;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      acc0[i] = o0[i];
      acc1[i] = o1[i];
    }
    return;
  }
  const FoldScale fA = fold_state(accA, segA);
  FoldScale fB = fA;
  if (kRowB) fB = fold_state(accB, segB);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {                      // registers i, i+1 belong to the same row
    if (!kRowB && (i & 2)) continue;
    const FoldScale f = (i & 2) ? fB : fA;
    const float2 r0 = fold_o2(make_float2(__uint_as_float(acc0[i]), __uint_as_float(acc0[i + 1])),
                              make_float2(__uint_as_float(o0[i]), __uint_as_float(o0[i + 1])), f);
    const float2 r1 = fold_o2(make_float2(__uint_as_float(acc1[i]), __uint_as_float(acc1[i + 1])),
                              make_float2(__uint_as_float(o1[i]), __uint_as_float(o1[i + 1])), f);
    acc0[i] = __float_as_uint(r0.x);
    acc0[i + 1] = __float_as_uint(r0.y);
    acc1[i] = __float_as_uint(r1.x);
    acc1[i + 1] = __float_as_uint(r1.y);
  }
}

}  // namespace kb
