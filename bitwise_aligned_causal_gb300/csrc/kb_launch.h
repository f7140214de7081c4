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
  uint32_t* err;    // device error word
};

struct DecodeArgs {
  const void* q;    // [B, Hq, 1, 128] bf16
  void* o;          // [B, Hq, 1, 128] bf16
  int B, Hq, Hkv;
  int ctx;          // keys 0..ctx-1 are visible; the query sits at ctx-1
  uint32_t* err;
};

// Query tiles per CTA of the prefill kernel: 1 (two CTAs per SM) or 2
// (two heads of one GQA group share every K/V tile).
cudaError_t launch_prefill(int q_tiles_per_cta, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_wait_probe(uint32_t* err, unsigned long long limit_ns, cudaStream_t s);

}  // namespace kb
