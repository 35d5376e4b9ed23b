// Kernel parameter blocks and launchers shared by the translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/lnk.h"

namespace lnk {

constexpr int kPage = 64;          // positions per page
constexpr int kBoxCols = 64;       // bf16 elements per TMA box row (128 bytes)
constexpr int kBoxBytes = kPage * kBoxCols * 2;  // one 64 x 64 bf16 box: 8 KiB
constexpr int kMaxDecodeRows = 4096;
constexpr int kMaxGroup = 8;

__host__ __device__ constexpr int boxes_for(int d) { return (d + kBoxCols - 1) / kBoxCols; }

// ---------------------------------------------------------------- append --
struct AppendParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* positions;
  const int32_t* rows;
  const int32_t* slots;
  const int32_t* table;
  const uint16_t* q_norm_w;
  const uint16_t* k_norm_w;
  uint16_t* k_pool;           // bf16 pools, or the 8-bit code pools when kv8 != 0
  uint16_t* v_pool;
  uint16_t* q_out;
  int32_t* status;
  double norm_eps;
  int T, hq, hkv, num_pages, num_rows, pages_per_row;
  int kv8;                    // pools hold E4M3 codes
  float k_scale, v_scale;     // their scales (a code c stands for e4m3(c) * scale)
  int splits;                 // CTAs per token (set by launch_append)
  float inv_freq[64];
};

cudaError_t launch_append(const AppendParams& p, int head_dim, cudaStream_t stream);

// ---------------------------------------------------------------- decode --
struct DecodeParams {
  const uint16_t* q;          // [B][Hq][D]
  const int32_t* positions;   // [B]
  const int32_t* table;       // [num_rows][pages_per_row]
  uint16_t* out;              // [B][Hq][D]
  int32_t* status;
  int32_t* ws_next;           // next chunk to claim (zero at rest)
  int32_t* ws_count;          // [B][Hkv] finished segments of cut pairs (zero at rest)
  float* ws_ml;               // [segments][G][2]: running max (log2 units), sum
  float* ws_o;                // [segments][G][D]: unnormalised partial outputs
  int B, hq, hkv, group, num_pages, pages_per_row, window;
  float scale_log2;           // softmax scale * log2(e) (8-bit pools: times the key scale)
  float out_scale;            // 1, or the value scale of an 8-bit pool
  // Fused decode step (fuse != 0): the CTA of pair (b, h) first rotates and
  // writes row b's token for kv head h (the append's work for that pair, with
  // `ap`: T = B, token b in table row b) and then attends.  Set only when every
  // pair is one CTA's single chunk.
  int fuse;
  AppendParams ap;
};

struct DecodeLaunch {
  int grid;        // persistent CTAs
  int smem_bytes;  // dynamic shared memory per CTA
  int mode;        // kernel variant (pool type, CTAs per SM)
};

// Workspace layout for `rows` decode rows and `grid` CTAs (byte offsets).
struct DecodeWorkspace {
  size_t next, count, ml, o, total;  // the counters (next, count) come first and must start at zero
};
constexpr int kChunksPerCta = 4;  // decode work chunks per persistent CTA
constexpr int kFuseMaxPages = 16;  // fused decode step: at most this many pages a (row, kv head) pair
DecodeWorkspace decode_workspace_layout(int rows, int hkv, int group, int head_dim, int grid);

// fused: the launch of the one-kernel decode step (two CTAs per SM when they fit)
cudaError_t decode_prepare(int head_dim, bool kv8, int B, int hkv, DecodeLaunch* launch, bool fused = false);

// lnk_paged_decode_attn with an option: clear_counters zeroes the workspace's
// counters on the stream once every argument check has passed, right before
// the launch (for a workspace whose previous contents are unknown).
lnk_status decode_entry(const lnk_attn_desc* desc, const lnk_bf16* q_roped, const int32_t* positions,
                        const int32_t* table, const lnk_bf16* k_pool, const lnk_bf16* v_pool, lnk_bf16* out,
                        int32_t B, void* workspace, size_t ws_bytes, int32_t* dev_status, lnk_stream stream,
                        bool clear_counters);
cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                          int head_dim, const DecodeLaunch& launch, cudaStream_t stream);

// ----------------------------------------------------------------- chunk --
// A chunk-attention CTA holds this many halves of 128 query rows.
constexpr int kChunkHalves = 2;

struct ChunkParams {
  const uint16_t* q;          // [P][Hq][D]
  const int32_t* rows;        // [P]
  const int32_t* positions;   // [P]
  const int32_t* segments;    // [P] or null
  const int32_t* table;
  uint16_t* out;              // [P][Hq][D]
  int32_t* status;
  int P, hq, hkv, group, num_pages, num_rows, pages_per_row, window;
  int tile_tokens, num_tiles;  // tokens per half tile (128 / group); tiles of kChunkHalves halves
  float scale_log2;
};

cudaError_t launch_chunk(const CUtensorMap& kmap, const CUtensorMap& vmap, const ChunkParams& p, int head_dim,
                         cudaStream_t stream);

// ------------------------------------------------------------ gather last --
cudaError_t launch_gather_last(const uint16_t* out, const int32_t* last, uint16_t* last_out, int M,
                               int P, int row_elems, int32_t* status, cudaStream_t stream);

// ------------------------------------------------------------- device info --
int device_sm_count();

// Host-side launch set-up, done once per device (and size) instead of per call.
cudaError_t set_max_dynamic_smem(const void* func, int bytes);
cudaError_t prefer_max_shared(const void* func);
cudaError_t occupancy_blocks(int* blocks, const void* func, int threads, size_t bytes);

}  // namespace lnk
