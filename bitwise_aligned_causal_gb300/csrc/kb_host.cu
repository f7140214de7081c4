// kb_host.cu -- the C ABI of libkb_attn.so: argument checks, TMA tensor-map
// encoding and kernel launches.  Declarations and their contract are in
// include/kb_attn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/kb_attn.h"
#include "kb_contract.cuh"
#include "kb_launch.h"

namespace {

constexpr int kMaxRows = 1 << 22;     // positions per sequence (4M)
constexpr int kMaxDevices = 64;

// Device error word (0 = fine).  Kernels get its address as an argument.
__device__ uint32_t g_kb_error_word;

// Library-owned scratch for kb_attn_decode_seg_static: the per-segment
// partials of a segmented decode (132 floats per row and segment), 4 MiB,
// one copy per device, reached through cudaGetSymbolAddress.
constexpr size_t kSegScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_seg_scratch[kSegScratchFloats];

struct DeviceState {
  uint32_t* err = nullptr;
  float* seg_scratch = nullptr;   // g_seg_scratch on this device
  int sm_count = 0;
  long long l2_bytes = 0;
  int cluster_fit[4] = {0, 0, 0, 0};   // clusters of 2, 4, 8 narrow packed CTAs the device runs at once
  bool ready = false;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

// Record a failed CUDA call for kb_attn_last_cuda_error and map it to a status.
kb_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = e;
  (void)cudaGetLastError();
  return KB_ERR_CUDA;
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

kb_status get_device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return KB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_kb_error_word)) != cudaSuccess) return cuda_fail(e);
    st.err = static_cast<uint32_t*>(p);
    if ((e = cudaGetSymbolAddress(&p, g_seg_scratch)) != cudaSuccess) return cuda_fail(e);
    st.seg_scratch = static_cast<float*>(p);
    if ((e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    int l2 = 0;
    if ((e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return cuda_fail(e);
    st.l2_bytes = l2;
    kb::packed_cluster_capacity(st.cluster_fit);
    st.ready = true;
  }
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q{};
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return KB_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = &st;
  return KB_OK;
}

// Key tiles of the busiest CTA under the tile kernel's snake schedule: units
// of n, n-1, ..., 1 key tiles (`per_len` units of each length), longest
// first, dealt to CTAs 0..G-1 and back.  The work is n * per_len steps.
long long snake_max_tiles(long long n, long long per_len, long long G) {
  static thread_local std::vector<long long> load;
  load.assign(static_cast<size_t>(G), 0);
  const long long units = n * per_len;
  for (long long i = 0; i < units; ++i) {
    const long long k = i / G, c = i % G;
    load[static_cast<size_t>((k & 1) ? G - 1 - c : c)] += n - i / per_len;
  }
  return *std::max_element(load.begin(), load.end());
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The pointer must be device (or managed) memory reachable from the current device.
kb_status check_device_pointer(const void* p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return KB_ERR_INVALID_ARG;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return KB_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KB_ERR_CUDA;
  if (attr.type == cudaMemoryTypeDevice && attr.device != dev) return KB_ERR_INVALID_ARG;
  return KB_OK;
}

// Rows of 128 bf16 seen as a 4-D tensor (64 columns, rows, 2 column halves,
// planes): the halves are 128 bytes apart inside a row, so one box of
// {64, 128, 2} moves a whole 128-row tile into the two 128-byte-swizzled
// slabs the MMA descriptors expect.  `rows` rows are in bounds in each of
// `planes` planes `plane_stride` bytes apart; reads beyond `rows` are
// zero-filled by the TMA unit.
kb_status encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t planes, uint64_t plane_stride) {
  cuuint64_t dims[4] = {64u, rows, 2u, planes};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kb::kHeadDim) * 2u, 128u, plane_stride};
  cuuint32_t box[4] = {64u, 128u, 2u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KB_OK : KB_ERR_CUDA;
}

kb_status check_heads(int B, int Hq, int Hkv) {
  if (B < 1 || Hq < 1 || Hkv < 1) return KB_ERR_INVALID_ARG;
  if (Hq != kb::kGroup * Hkv) return KB_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > (1LL << 24)) return KB_ERR_UNSUPPORTED;
  return KB_OK;
}

kb_status check_ptrs(const void* q, const void* k, const void* v, const void* o) {
  if (!q || !k || !v || !o) return KB_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return KB_ERR_INVALID_ARG;
  return KB_OK;
}

// A paged K/V pool [num_pages, Hkv, page_size, 128] and its page table.
struct Paging {
  const int* block_table = nullptr;  // device [B, pages_per_seq]
  int pages_per_seq = 0, page_size = 0, num_pages = 0;
};

kb_status check_paging(const Paging& pg, int Hkv) {
  if (!pg.block_table || (reinterpret_cast<uintptr_t>(pg.block_table) & 3u)) return KB_ERR_INVALID_ARG;
  if (pg.pages_per_seq < 1 || pg.num_pages < 1 || pg.page_size < kb::kTileKeys) return KB_ERR_INVALID_ARG;
  if (pg.page_size % kb::kTileKeys != 0) return KB_ERR_UNSUPPORTED;
  if (static_cast<long long>(pg.pages_per_seq) * pg.page_size > kMaxRows) return KB_ERR_UNSUPPORTED;
  if (static_cast<long long>(pg.num_pages) * Hkv > 0x7FFFFFFFLL) return KB_ERR_UNSUPPORTED;
  return KB_OK;
}

// Per-sequence start positions and row counts of a ragged batch (device arrays).
struct Ragged {
  const int* starts = nullptr;
  const int* lens = nullptr;
};

// CTAs per (sub-chunk, b, kv head) of the packed kernel's fold mode: the
// largest cluster whose clusters all run at once (one wave), when the batch
// alone would leave SMs idle.  Narrow rows only; the other CTAs of a cluster
// keep their segments' partials in shared memory, so a CTA may own at most
// as many segments as it has partial slots.
int choose_cluster(const DeviceState& dst, int L, int n_sub, int B, int Hkv, int n_kv_max) {
  if (L > 2) return 1;
  const long long units = static_cast<long long>(n_sub) * B * Hkv;
  if (2 * units > dst.sm_count) return 1;
  const int ns = (n_kv_max + kb::kSegTiles - 1) / kb::kSegTiles;
  const long long slots = kb::packed_partial_slots(kb::kGroup * L);
  for (int i = 3, c = 8; i >= 1; --i, c /= 2) {
    if (c > ns || units > dst.cluster_fit[i]) continue;
    if ((ns + c - 1) / c > slots) continue;
    return c;
  }
  return 1;
}

// seg_tiles: 0 for the default entry points (the contract's segment length,
// folded in the kernels); > 0 for the *_seg entry points (that length; chunks
// of at most 32 rows then leave per-segment partials in `workspace`, which a
// second kernel folds).
kb_status chunk_impl(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int L, int start,
                     int kv_cap, int cta_shape, void* stream, const Paging* paging = nullptr,
                     const Ragged* ragged = nullptr, float* lse = nullptr, int seg_tiles = 0,
                     void* workspace = nullptr, size_t workspace_bytes = 0) {
  kb_status s = check_ptrs(q, k, v, o);
  if (s != KB_OK) return s;
  if ((s = check_heads(B, Hq, Hkv)) != KB_OK) return s;
  if (L < 1 || start < 0 || kv_cap < 1) return KB_ERR_INVALID_ARG;
  if (static_cast<long long>(start) + L > kv_cap) return KB_ERR_INVALID_ARG;
  if (kv_cap > kMaxRows) return KB_ERR_UNSUPPORTED;
  if (cta_shape != 0 && cta_shape != kb::kShapeOneTilePerSm && cta_shape != kb::kShapePersistent &&
      cta_shape != kb::kShapeSnake)
    return KB_ERR_INVALID_ARG;
  const bool force_persistent = (cta_shape == kb::kShapePersistent);
  const bool force_snake = (cta_shape == kb::kShapeSnake);
  const bool packed = (cta_shape == 0);
  if (packed && L > kb::kMaxPackedRows) return KB_ERR_INVALID_ARG;
  if (lse != nullptr && packed) return KB_ERR_INVALID_ARG;
  if (seg_tiles < 0) return KB_ERR_INVALID_ARG;
  const bool explicit_seg = seg_tiles > 0;
  if (explicit_seg) {
    // the *_seg entry points: contiguous caches, no log-sum-exp; short chunks
    // leave their per-segment partials in the caller's workspace
    if (paging || ragged || lse) return KB_ERR_UNSUPPORTED;
    if (packed) {
      const int n_kv = (start + L - 1) / kb::kTileKeys + 1;
      const long long n_seg = (n_kv + seg_tiles - 1) / seg_tiles;
      const unsigned long long need =
          static_cast<unsigned long long>(B) * Hq * L * n_seg * kb::kPartFloats * sizeof(float);
      if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return KB_ERR_INVALID_ARG;
      if (n_seg * 2LL * B * Hkv > 0x7FFFFFFFLL) return KB_ERR_UNSUPPORTED;
    }
  }
  const int seg = explicit_seg ? seg_tiles : kb::kSegTiles;
  // a ragged batch sizes the grid for its longest possible sequence
  const int first_tile = ragged ? 0 : start / kb::kTileRows;
  const int last_tile = ragged ? (L + kb::kTileRows - 2) / kb::kTileRows : (start + L - 1) / kb::kTileRows;
  // CTAs: the tile kernel at most one per (query tile, batch, head); the
  // packed kernel at most two sub-chunks x a cluster of 8 per (batch, KV head)
  const long long grid = !packed ? static_cast<long long>(last_tile - first_tile + 1) * B * Hq : 16LL * B * Hkv;
  if (grid > 0x7FFFFFFFLL) return KB_ERR_UNSUPPORTED;

  DeviceState* dst = nullptr;
  if ((s = get_device_state(&dst)) != KB_OK) return s;
  for (const void* p : {q, k, v, static_cast<const void*>(o)})
    if ((s = check_device_pointer(p)) != KB_OK) return s;
  if (paging && (s = check_device_pointer(paging->block_table)) != KB_OK) return s;
  if (lse && (s = check_device_pointer(lse)) != KB_OK) return s;
  if (ragged) {
    if ((s = check_device_pointer(ragged->starts)) != KB_OK) return s;
    if ((s = check_device_pointer(ragged->lens)) != KB_OK) return s;
  }

  CUtensorMap tq, tk, tv;
  const uint64_t row_bytes = kb::kHeadDim * 2u;
  // a contiguous uniform batch ends its K/V map at the chunk's last key; a
  // ragged batch maps the whole cache (the kernels zero V rows past each sequence)
  const uint64_t kv_len = ragged ? static_cast<uint64_t>(kv_cap) : static_cast<uint64_t>(start) + L;
  // K/V maps: a contiguous cache ends at the chunk's last key (later rows read
  // as zeros); a paged pool is [num_pages * Hkv planes, page_size rows].
  const uint64_t kv_rows = paging ? static_cast<uint64_t>(paging->page_size) : kv_len;
  const uint64_t kv_planes =
      paging ? static_cast<uint64_t>(paging->num_pages) * Hkv : static_cast<uint64_t>(B) * Hkv;
  const uint64_t kv_stride = (paging ? static_cast<uint64_t>(paging->page_size) : static_cast<uint64_t>(kv_cap)) *
                             row_bytes;
  if ((s = encode_rows_map(&tk, k, kv_rows, kv_planes, kv_stride)) != KB_OK) return s;
  if ((s = encode_rows_map(&tv, v, kv_rows, kv_planes, kv_stride)) != KB_OK) return s;
  if (packed) {
    // query rows packed by GQA group
    const int split = std::min(L, kb::kTileKeys - start % kb::kTileKeys);
    const int n_sub = (ragged || split < L) ? 2 : 1;
    kb::PackedArgs a{};
    a.q = q;
    a.o = o;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.L = L;
    a.start = start;
    a.max_ctx = kv_cap;
    if (ragged) {
      a.starts = ragged->starts;
      a.lens = ragged->lens;
    }
    if (paging) {
      a.block_table = paging->block_table;
      a.pages_per_seq = paging->pages_per_seq;
      a.page_size = paging->page_size;
      a.num_pages = paging->num_pages;
    }
    a.err = dst->err;
    a.n_sub = n_sub;
    int n_seg = 0;
    if (explicit_seg) {
      const int n_kv = (start + L - 1) / kb::kTileKeys + 1;
      n_seg = (n_kv + seg - 1) / seg;
      if ((s = check_device_pointer(workspace)) != KB_OK) return s;
      a.seg_tiles = seg;
      a.n_seg = n_seg;
      a.part = static_cast<float*>(workspace);
    } else {
      const int n_kv_max = ragged ? (kv_cap - 1) / kb::kTileKeys + 1 : (start + L - 1) / kb::kTileKeys + 1;
      a.fold_seg = seg;
      a.cluster = choose_cluster(*dst, L, n_sub, B, Hkv, n_kv_max);
    }
    cudaError_t e = kb::launch_packed(tk, tv, a, n_sub, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess && explicit_seg)
      e = kb::launch_seg_fold(static_cast<const float*>(workspace), o, static_cast<long long>(B) * Hq * L, L, start,
                              seg, n_seg, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return KB_OK;
  }
  if ((s = encode_rows_map(&tq, q, static_cast<uint64_t>(L), static_cast<uint64_t>(B) * Hq,
                           static_cast<uint64_t>(L) * row_bytes)) != KB_OK)
    return s;

  kb::PrefillArgs a{};
  a.o = o;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.L = L;
  a.start = start;
  a.first_tile = first_tile;
  a.n_tiles = last_tile - first_tile + 1;
  a.kv_cap = kv_cap;
  // beyond a few waves, order CTAs by GQA group so that the resident ones
  // share K/V in L2; below that, globally longest tile first
  a.group_major = grid > 4LL * dst->sm_count ? 1 : 0;
  a.lse = lse;
  a.seg_tiles = seg;
  a.max_ctas = dst->sm_count > 0 ? dst->sm_count : 1;
  {
    // Persistent when what it saves beats what it costs: it hides a CTA's
    // start and end (about 5000 cycles, fitted to timings of both launches
    // from S=1.5K to 16K) under the previous unit, against a unit of (n+1)/2
    // key tiles at about 1550 cycles each; its static split leaves a tail of
    // (ceil(p) - p) / p with p pairs per CTA, where the one-CTA-per-tile
    // launch ends on the shortest tiles.
    const long long pairs = static_cast<long long>((a.n_tiles + 1) / 2) * kb::kGroup * B * Hkv;
    bool persistent = pairs <= a.max_ctas;
    if (!persistent) {
      const double p = static_cast<double>(pairs) / a.max_ctas;
      const double tail = (std::ceil(p) - p) / p;
      const double saved = 5000.0 / (0.5 * (a.n_tiles + 1) * 1550.0 + 5000.0);
      persistent = saved > tail;
    }
    a.persistent = (force_persistent || persistent) ? kb::kSchedPairs : kb::kSchedOnePerCta;
    // The snake, when it balances better than the pairs (few pairs per CTA)
    // and all of K and V fit in three quarters of L2: it runs every group at
    // once.
    const long long kv_bytes = 2LL * B * Hkv * (start + L) * kb::kHeadDim * 2;
    if (force_snake) {
      a.persistent = kb::kSchedSnake;
    } else if (!force_persistent && !ragged && 4 * kv_bytes <= 3 * dst->l2_bytes &&
               pairs < 32LL * a.max_ctas) {
      const long long n = a.n_tiles, G = a.max_ctas;
      const long long units = n * B * Hq;
      const long long per_cta_pairs = (pairs + G - 1) / G;
      double est = a.persistent == kb::kSchedPairs
                       ? per_cta_pairs * (n + 1) * 1550.0 + 5000.0
                       : (static_cast<double>(units) * 5000.0 + 0.5 * n * (n + 1) * B * Hq * 1550.0) / G;
      const long long snake_tiles = snake_max_tiles(n, static_cast<long long>(B) * Hq, G);
      if (snake_tiles * 1550.0 + 5000.0 < est) a.persistent = kb::kSchedSnake;
    }
  }
  if (ragged) {
    a.starts = ragged->starts;
    a.lens = ragged->lens;
  }
  if (paging) {
    a.block_table = paging->block_table;
    a.pages_per_seq = paging->pages_per_seq;
    a.page_size = paging->page_size;
    a.num_pages = paging->num_pages;
  }
  a.err = dst->err;
  const cudaError_t e = kb::launch_prefill_s2(tq, tk, tv, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KB_OK;
}

constexpr int kDefaultQTilesPerCta = kb::kShapeOneTilePerSm;

// Chunks of at most this many query rows go to the packed kernel.
int chunk_cta_shape(int L) { return L <= kb::kMaxPackedRows ? 0 : kDefaultQTilesPerCta; }

}  // namespace

extern "C" {

kb_status kb_attn_chunk(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int L,
                        int start, int kv_cap, void* stream) {
  return chunk_impl(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, chunk_cta_shape(L), stream);
}

kb_status kb_attn_chunk_cta_shape(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                                  int L, int start, int kv_cap, int q_tiles_per_cta, void* stream) {
  return chunk_impl(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, q_tiles_per_cta, stream);
}

kb_status kb_attn_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int S,
                          void* stream) {
  if (S < 1) return KB_ERR_INVALID_ARG;
  return chunk_impl(q, k, v, o, B, Hq, Hkv, S, 0, S, chunk_cta_shape(S), stream);
}

kb_status kb_attn_prefill_seg(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int S,
                              int seg_tiles, void* stream) {
  if (S < 1 || seg_tiles < 1) return KB_ERR_INVALID_ARG;
  return chunk_impl(q, k, v, o, B, Hq, Hkv, S, 0, S, kb::kShapeOneTilePerSm, stream, nullptr, nullptr, nullptr,
                    seg_tiles);
}

size_t kb_attn_seg_workspace_bytes(int B, int Hq, int L, int start, int seg_tiles) {
  if (B < 1 || Hq < 1 || L < 1 || start < 0 || seg_tiles < 1 || L > kb::kMaxPackedRows) return 0;
  const int n_kv = (start + L - 1) / kb::kTileKeys + 1;
  const int n_seg = (n_kv + seg_tiles - 1) / seg_tiles;
  return static_cast<size_t>(B) * Hq * L * n_seg * kb::kPartFloats * sizeof(float);
}

kb_status kb_attn_chunk_seg(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int L,
                            int start, int kv_cap, int seg_tiles, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (seg_tiles < 1) return KB_ERR_INVALID_ARG;
  return chunk_impl(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, chunk_cta_shape(L), stream, nullptr, nullptr, nullptr,
                    seg_tiles, workspace, workspace_bytes);
}

kb_status kb_attn_decode_seg(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                             int ctx_len, int kv_cap, int seg_tiles, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (ctx_len < 1 || ctx_len > kv_cap || seg_tiles < 1) return KB_ERR_INVALID_ARG;
  return chunk_impl(q, k, v, o, B, Hq, Hkv, 1, ctx_len - 1, kv_cap, 0, stream, nullptr, nullptr, nullptr, seg_tiles,
                    workspace, workspace_bytes);
}

kb_status kb_attn_decode_seg_static(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                                    int ctx_len, int kv_cap, int seg_tiles, void* stream) {
  // the argument checks every entry point makes come first, so a bad
  // pointer or head count gets the same status here as elsewhere
  kb_status s = check_ptrs(q, k, v, o);
  if (s != KB_OK) return s;
  if ((s = check_heads(B, Hq, Hkv)) != KB_OK) return s;
  if (ctx_len < 1 || ctx_len > kv_cap || seg_tiles < 1) return KB_ERR_INVALID_ARG;
  const size_t need = kb_attn_seg_workspace_bytes(B, Hq, 1, ctx_len - 1, seg_tiles);
  if (need == 0) return KB_ERR_INVALID_ARG;
  if (need > kSegScratchFloats * sizeof(float)) return KB_ERR_UNSUPPORTED;
  DeviceState* dst = nullptr;
  if ((s = get_device_state(&dst)) != KB_OK) return s;
  return chunk_impl(q, k, v, o, B, Hq, Hkv, 1, ctx_len - 1, kv_cap, 0, stream, nullptr, nullptr, nullptr, seg_tiles,
                    dst->seg_scratch, kSegScratchFloats * sizeof(float));
}

kb_status kb_attn_prefill_lse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                              int Hkv, int S, void* stream) {
  if (S < 1 || lse == nullptr) return KB_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return KB_ERR_INVALID_ARG;
  return chunk_impl(q, k, v, o, B, Hq, Hkv, S, 0, S, kb::kShapeOneTilePerSm, stream, nullptr, nullptr, lse);
}

kb_status kb_attn_backward(const void* q, const void* k, const void* v, const void* o, const void* dout,
                           const float* lse, float* delta, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                           int S, void* stream) {
  kb_status s = check_ptrs(q, k, v, o);
  if (s != KB_OK) return s;
  if ((s = check_ptrs(dout, dq, dk, dv)) != KB_OK) return s;
  if (!lse || !delta || (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(delta) & 3u))
    return KB_ERR_INVALID_ARG;
  if ((s = check_heads(B, Hq, Hkv)) != KB_OK) return s;
  if (S < 1) return KB_ERR_INVALID_ARG;
  if (S > kMaxRows) return KB_ERR_UNSUPPORTED;
  const int n_tiles = (S + kb::kTileRows - 1) / kb::kTileRows;
  if (static_cast<long long>(n_tiles) * B * Hq > 0x7FFFFFFFLL) return KB_ERR_UNSUPPORTED;
  DeviceState* dst = nullptr;
  if ((s = get_device_state(&dst)) != KB_OK) return s;
  for (const void* p : {q, k, v, o, dout, static_cast<const void*>(lse), static_cast<const void*>(delta),
                        static_cast<const void*>(dq), static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if ((s = check_device_pointer(p)) != KB_OK) return s;
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t row_bytes = kb::kHeadDim * 2u;
  const uint64_t rows = static_cast<uint64_t>(S);
  if ((s = encode_rows_map(&tq, q, rows, static_cast<uint64_t>(B) * Hq, rows * row_bytes)) != KB_OK) return s;
  if ((s = encode_rows_map(&tdo, dout, rows, static_cast<uint64_t>(B) * Hq, rows * row_bytes)) != KB_OK) return s;
  if ((s = encode_rows_map(&tk, k, rows, static_cast<uint64_t>(B) * Hkv, rows * row_bytes)) != KB_OK) return s;
  if ((s = encode_rows_map(&tv, v, rows, static_cast<uint64_t>(B) * Hkv, rows * row_bytes)) != KB_OK) return s;
  kb::BwdArgs a{};
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.delta = delta;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.S = S;
  a.n_tiles = n_tiles;
  a.group_major = static_cast<long long>(n_tiles) * B * Hq > 4LL * dst->sm_count ? 1 : 0;
  a.err = dst->err;
  const cudaError_t e = kb::launch_backward(tq, tk, tv, tdo, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KB_OK;
}

kb_status kb_attn_chunk_paged(const void* q, const void* k_pages, const void* v_pages, void* o, int B, int Hq,
                              int Hkv, int L, int start, const int* block_table, int pages_per_seq, int page_size,
                              int num_pages, void* stream) {
  Paging pg;
  pg.block_table = block_table;
  pg.pages_per_seq = pages_per_seq;
  pg.page_size = page_size;
  pg.num_pages = num_pages;
  kb_status s = check_heads(B, Hq, Hkv);
  if (s != KB_OK) return s;
  if ((s = check_paging(pg, Hkv)) != KB_OK) return s;
  const long long cap = static_cast<long long>(pages_per_seq) * page_size;
  return chunk_impl(q, k_pages, v_pages, o, B, Hq, Hkv, L, start, static_cast<int>(cap), chunk_cta_shape(L), stream,
                    &pg);
}

kb_status kb_attn_chunk_varlen(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                               int L_max, const int* starts, const int* lens, int kv_cap, const int* block_table,
                               int pages_per_seq, int page_size, int num_pages, void* stream) {
  kb_status s = check_heads(B, Hq, Hkv);
  if (s != KB_OK) return s;
  if (!starts || !lens || (reinterpret_cast<uintptr_t>(starts) & 3u) || (reinterpret_cast<uintptr_t>(lens) & 3u))
    return KB_ERR_INVALID_ARG;
  Ragged rg;
  rg.starts = starts;
  rg.lens = lens;
  if (block_table) {
    Paging pg;
    pg.block_table = block_table;
    pg.pages_per_seq = pages_per_seq;
    pg.page_size = page_size;
    pg.num_pages = num_pages;
    if ((s = check_paging(pg, Hkv)) != KB_OK) return s;
    const int cap = pages_per_seq * page_size;
    if (L_max < 1 || L_max > cap) return KB_ERR_INVALID_ARG;
    return chunk_impl(q, k, v, o, B, Hq, Hkv, L_max, 0, cap, chunk_cta_shape(L_max), stream, &pg, &rg);
  }
  if (L_max < 1 || kv_cap < 1 || L_max > kv_cap) return KB_ERR_INVALID_ARG;
  return chunk_impl(q, k, v, o, B, Hq, Hkv, L_max, 0, kv_cap, chunk_cta_shape(L_max), stream, nullptr, &rg);
}

kb_status kb_attn_decode(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int ctx_len,
                         int kv_cap, void* stream) {
  kb_status s = check_ptrs(q, k, v, o);
  if (s != KB_OK) return s;
  if ((s = check_heads(B, Hq, Hkv)) != KB_OK) return s;
  if (ctx_len < 1 || kv_cap < 1 || ctx_len > kv_cap) return KB_ERR_INVALID_ARG;
  if (kv_cap > kMaxRows) return KB_ERR_UNSUPPORTED;
  // one query row at position ctx_len - 1: the packed chunk path with L = 1
  return chunk_impl(q, k, v, o, B, Hq, Hkv, 1, ctx_len - 1, kv_cap, 0, stream);
}

kb_status kb_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o, int B, int Hq,
                               int Hkv, const int* block_table, int pages_per_seq, int page_size, int num_pages,
                               const int* ctx_lens, void* stream) {
  kb_status s = check_ptrs(q, k_pages, v_pages, o);
  if (s != KB_OK) return s;
  if ((s = check_heads(B, Hq, Hkv)) != KB_OK) return s;
  if (!ctx_lens || (reinterpret_cast<uintptr_t>(ctx_lens) & 3u)) return KB_ERR_INVALID_ARG;
  Paging pg;
  pg.block_table = block_table;
  pg.pages_per_seq = pages_per_seq;
  pg.page_size = page_size;
  pg.num_pages = num_pages;
  if ((s = check_paging(pg, Hkv)) != KB_OK) return s;

  DeviceState* dst = nullptr;
  if ((s = get_device_state(&dst)) != KB_OK) return s;
  for (const void* p : {q, k_pages, v_pages, static_cast<const void*>(o), static_cast<const void*>(block_table),
                        static_cast<const void*>(ctx_lens)})
    if ((s = check_device_pointer(p)) != KB_OK) return s;

  // pools [num_pages, Hkv, page_size, 128]: plane = page * Hkv + kv head
  CUtensorMap tk, tv;
  const uint64_t row_bytes = kb::kHeadDim * 2u;
  const uint64_t planes = static_cast<uint64_t>(num_pages) * Hkv;
  if ((s = encode_rows_map(&tk, k_pages, static_cast<uint64_t>(page_size), planes,
                           static_cast<uint64_t>(page_size) * row_bytes)) != KB_OK)
    return s;
  if ((s = encode_rows_map(&tv, v_pages, static_cast<uint64_t>(page_size), planes,
                           static_cast<uint64_t>(page_size) * row_bytes)) != KB_OK)
    return s;
  kb::PackedArgs a{};
  a.q = q;
  a.o = o;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.L = 1;
  a.ctx_lens = ctx_lens;
  a.max_ctx = pages_per_seq * page_size;
  a.fold_seg = kb::kSegTiles;
  a.cluster = choose_cluster(*dst, 1, 1, B, Hkv, (a.max_ctx - 1) / kb::kTileKeys + 1);
  a.block_table = block_table;
  a.pages_per_seq = pages_per_seq;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.err = dst->err;
  const cudaError_t e = kb::launch_packed(tk, tv, a, 1, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KB_OK;
}

kb_status kb_attn_check_device_status(void* stream) {
  DeviceState* dst = nullptr;
  kb_status s = get_device_state(&dst);
  if (s != KB_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t word = 0;
  if ((e = cudaMemcpy(&word, dst->err, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpy(dst->err, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess) return cuda_fail(e);
    return word >= kb::kDevBadInput ? KB_ERR_INVALID_ARG : KB_ERR_TIMEOUT;
  }
  return KB_OK;
}

kb_status kb_attn_debug_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return KB_ERR_INVALID_ARG;
  DeviceState* dst = nullptr;
  kb_status s = get_device_state(&dst);
  if (s != KB_OK) return s;
  const cudaError_t e = kb::launch_wait_probe(dst->err, static_cast<unsigned long long>(limit_us) * 1000ull,
                                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KB_OK;
}

const char* kb_status_string(kb_status s) {
  switch (s) {
    case KB_OK: return "ok";
    case KB_ERR_INVALID_ARG: return "invalid argument";
    case KB_ERR_UNSUPPORTED: return "shape outside the numerical contract";
    case KB_ERR_CUDA: return "CUDA call failed";
    case KB_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int kb_contract_version(void) { return kb::kContractVersion; }

int kb_attn_last_cuda_error(void) { return static_cast<int>(t_last_cuda_error); }

const char* kb_attn_last_cuda_error_string(void) { return cudaGetErrorString(t_last_cuda_error); }

}  // extern "C"
