// kb_segment.cu -- the fold of the C5 segmented mode for the packed kernel.
//
// In segmented mode the packed kernel (decode and chunks of at most 32 rows)
// runs one CTA per (segment, sub-chunk, b, kv head) and leaves each row's
// per-segment partial (O unnormalised, m, mc, l) in the caller's workspace.
// This kernel folds a row's segments left to right with fold_state / fold_o
// (the functions the segmented tile kernel applies in TMEM at its segment
// ends) and normalises (C4), so every entry point of the mode gives the same
// bits (KernelBraid README, "Method": one contract for prefill, partitioned
// forward and decode).
#include "kb_contract.cuh"
#include "kb_launch.h"

namespace kb {

// One warp per output row (b, h, r): lane l owns columns 4l..4l+3.
__global__ void __launch_bounds__(256) kb_seg_fold_kernel(const float* __restrict__ part,
                                                          __nv_bfloat16* __restrict__ o, long long rows, int L,
                                                          int start, int seg_tiles, int n_seg) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int r = static_cast<int>(row % L);
  const int n_kv = (start + r) / kTileKeys + 1;                   // C1: tiles 0..floor(p / 128)
  const int ns = (n_kv + seg_tiles - 1) / seg_tiles;              // this row's segments
  const float* p = part + static_cast<size_t>(row) * n_seg * kPartFloats;
  float4 acc_o = reinterpret_cast<const float4*>(p)[lane];        // segment 0 as it is
  const float4 s0 = reinterpret_cast<const float4*>(p + 128)[0];
  RowState acc{s0.x, s0.y, s0.z};
  for (int sg = 1; sg < ns; ++sg) {
    const float* q = p + static_cast<size_t>(sg) * kPartFloats;
    const float4 so = reinterpret_cast<const float4*>(q)[lane];
    const float4 st = reinterpret_cast<const float4*>(q + 128)[0];
    const RowState seg{st.x, st.y, st.z};
    const FoldScale f = fold_state(acc, seg);
    acc_o.x = fold_o(acc_o.x, so.x, f);
    acc_o.y = fold_o(acc_o.y, so.y, f);
    acc_o.z = fold_o(acc_o.z, so.z, f);
    acc_o.w = fold_o(acc_o.w, so.w, f);
  }
  const float inv_l = row_inv_l(acc);
  uint2 w;
  w.x = pack_bf16x2(__fmul_rn(acc_o.x, inv_l), __fmul_rn(acc_o.y, inv_l));
  w.y = pack_bf16x2(__fmul_rn(acc_o.z, inv_l), __fmul_rn(acc_o.w, inv_l));
  reinterpret_cast<uint2*>(o + static_cast<size_t>(row) * kHeadDim)[lane] = w;
}

cudaError_t launch_seg_fold(const float* part, void* o, long long rows, int L, int start, int seg_tiles, int n_seg,
                            cudaStream_t s) {
  kb_seg_fold_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(
      part, static_cast<__nv_bfloat16*>(o), rows, L, start, seg_tiles, n_seg);
  return cudaGetLastError();
}

}  // namespace kb
