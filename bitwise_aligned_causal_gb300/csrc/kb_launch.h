// kb_launch.h -- host-side launchers of the attention kernels (internal; the
// public C ABI is include/kb_attn.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace kb {

struct PrefillArgs {
  void* o;          // [B, Hq, L, 128] bf16 output rows start..start+L-1
  int B, Hq, Hkv;
  int L;            // query rows in this call
  int start;        // absolute position of query row 0
  int first_tile;   // floor(start / 128)
  int n_tiles;      // absolute query tiles touched by [start, start+L)
  const int* block_table;  // optional device [B, pages_per_seq]: paged K/V pools
  int pages_per_seq, page_size, num_pages;
  const int* starts;       // optional device [B]: per-sequence start (ragged batch; then
  const int* lens;         //   L is the row stride of q and o and lens[b] <= L rows are used)
  int kv_cap;              // keys per sequence the cache can hold
  int group_major;         // CTA order: 1 = (b, g) slowest, 0 = query tile slowest
  float* lse;              // optional [B, Hq, L] fp32: natural-log log-sum-exp of each row's scaled scores
  int seg_tiles;           // C5 segment length in key tiles (0: the whole row is one segment)
  int max_ctas;            // CTAs of a persistent launch (one per SM)
  int persistent;          // schedule: kSchedOnePerCta, kSchedPairs or kSchedSnake
  uint32_t* err;    // device error word
};

// Query rows packed by GQA group (decode and chunks of at most 32 rows).
struct PackedArgs {
  const void* q;           // [B, Hq, L, 128] bf16
  void* o;                 // [B, Hq, L, 128] bf16
  int B, Hq, Hkv;
  int L;                   // query rows per (batch, head)
  int start;               // absolute position of query row 0 (when ctx_lens is null)
  const int* ctx_lens;     // optional device [B]: row L-1 of batch b sits at ctx_lens[b] - 1
  int max_ctx;             // largest valid ctx_lens entry (cache capacity)
  const int* block_table;  // optional device [B, pages_per_seq]: paged K/V pools
  int pages_per_seq, page_size, num_pages;
  const int* starts;       // optional device [B]: per-sequence start and row count (ragged
  const int* lens;         //   batch); L is then the row stride of q and o
  int n_sub;               // sub-chunks per (b, kv head) in the grid (1 or 2)
  // fold mode (part == nullptr): C5 segments of fold_seg key tiles, cut into
  // contiguous blocks over a cluster of `cluster` CTAs per (sub, b, g); the
  // cluster's first CTA folds them all and writes o
  int fold_seg, cluster;
  // workspace mode (part != nullptr): CTA (seg, sub, b, g) runs key tiles
  // [seg * seg_tiles, +seg_tiles) from the fresh state and writes the rows'
  // partial (O[128], m, mc, l) to part[((b*Hq + h)*L + r)*n_seg + seg][132]
  int seg_tiles, n_seg;
  float* part;
  uint32_t* err;
};

constexpr int kPartFloats = 132;   // one partial: O[128], m, mc, l, pad

constexpr int kMaxPackedRows = 32;   // query rows per (batch, head) the packed kernel takes

// One 128-row query tile per CTA, one CTA per SM, three S buffers in TMEM
// and separate Q K^T / P V issuers, so the tensor pipe works on later key
// tiles while the softmax runs (CTA shape 3).
constexpr int kShapeOneTilePerSm = 3;
// The same kernel with the persistent launch forced (tests of the schedule):
// 4 with pairs of query tiles, 5 with the snake.
constexpr int kShapePersistent = 4;
constexpr int kShapeSnake = 5;
// The tile kernel's schedules (PrefillArgs::persistent).
constexpr int kSchedOnePerCta = 0;   // one CTA per unit
constexpr int kSchedPairs = 1;       // persistent, balanced pairs of query tiles, group-major
constexpr int kSchedSnake = 2;       // persistent, single units longest first, dealt back and forth
cudaError_t launch_prefill_s2(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const PrefillArgs& a, cudaStream_t s);
// n_sub: 1, or 2 when the chunk crosses a 128-position tile boundary.
cudaError_t launch_packed(const CUtensorMap& tk, const CUtensorMap& tv, const PackedArgs& a, int n_sub,
                          cudaStream_t s);
// Partials a CTA of the narrow packed kernel can keep in shared memory for
// the cluster's first CTA, with n_rows packed rows.
uint32_t packed_partial_slots(int n_rows);
// Clusters of 2, 4 and 8 CTAs (entries 1, 2, 3) of the narrow packed kernel
// the current device runs at once; entry 0 is unused.
void packed_cluster_capacity(int (&active)[4]);
// Gradient of a whole-sequence causal prefill (query row i at position i).
struct BwdArgs {
  const void* o;           // [B, Hq, S, 128] bf16 forward output
  const void* dout;        // [B, Hq, S, 128] bf16 gradient of the output
  const float* lse;        // [B, Hq, S] natural-log log-sum-exp from the forward
  float* delta;            // [B, Hq, S] out: rowsum(dout * o)
  void* dq;                // [B, Hq, S, 128] bf16 out
  void* dk;                // [B, Hkv, S, 128] bf16 out
  void* dv;                // [B, Hkv, S, 128] bf16 out
  int B, Hq, Hkv, S;
  int n_tiles;             // ceil(S / 128)
  int group_major;         // CTA order of the dq kernel (as PrefillArgs)
  uint32_t* err;
};
// delta, then dq (query-major), then dk/dv (key-major), all on stream s.
// tq, tdo: [B*Hq planes, S rows]; tk, tv: [B*Hkv planes, S rows].
cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t s);
// C5 fold of the packed kernel's per-segment partials, one warp per row
// (rows = B*Hq*L, row r of a (b, h) at position start + r), then C4 into o.
cudaError_t launch_seg_fold(const float* part, void* o, long long rows, int L, int start, int seg_tiles, int n_seg,
                            cudaStream_t s);
cudaError_t launch_wait_probe(uint32_t* err, unsigned long long limit_ns, cudaStream_t s);

}  // namespace kb
