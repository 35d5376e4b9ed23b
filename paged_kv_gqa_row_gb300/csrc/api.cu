// C ABI entry points of liblnk: argument checks, frequency tables, tensor
// maps and launches.  Nothing here allocates device memory or synchronises.
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>

#include "common.cuh"

namespace lnk {

namespace {

constexpr int kMaxDevices = 64;

int g_sm_count[kMaxDevices];
std::once_flag g_sm_once[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Tensor map over one pool: rows = kv_heads * num_pages * 64 positions, each
// head_dim bf16 wide; boxes of 64 positions x 64 elements, 128-byte swizzle.
bool make_pool_map(CUtensorMap* map, const void* pool, const lnk_attn_desc& d) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  // 8-bit pools are viewed as 16-bit pairs: a page row of D codes is D / 2
  // elements, so one 64 x 64 box (128-byte rows) covers a whole page
  const bool kv8 = d.kv_dtype == LNK_KV_E4M3;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kv8 ? d.head_dim / 2 : d.head_dim),
                        static_cast<cuuint64_t>(d.num_kv_heads) * d.num_pages * kPage};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * (kv8 ? 1 : 2)};
  cuuint32_t box[2] = {kBoxCols, kPage};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// make_pool_map with a small per-thread cache: a serving loop passes the same
// pools every step, and encoding a tensor map costs microseconds of host time.
bool pool_map(CUtensorMap* map, const void* pool, const lnk_attn_desc& d) {
  struct Entry {
    const void* pool = nullptr;
    int head_dim = 0, num_kv_heads = 0, num_pages = 0, kv_dtype = 0;
    CUtensorMap map;
  };
  thread_local Entry cache[4];
  thread_local int next = 0;
  for (const Entry& e : cache)
    if (e.pool == pool && e.head_dim == d.head_dim && e.num_kv_heads == d.num_kv_heads &&
        e.num_pages == d.num_pages && e.kv_dtype == d.kv_dtype) {
      *map = e.map;
      return true;
    }
  if (!make_pool_map(map, pool, d)) return false;
  Entry& e = cache[next];
  next = (next + 1) % 4;
  e.pool = pool;
  e.head_dim = d.head_dim;
  e.num_kv_heads = d.num_kv_heads;
  e.num_pages = d.num_pages;
  e.kv_dtype = d.kv_dtype;
  e.map = *map;
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks shared by every entry point.
lnk_status check_desc(const lnk_attn_desc* d) {
  if (d == nullptr) return LNK_EINVAL;
  if (d->page_size != kPage) return LNK_EUNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 96 && d->head_dim != 128) return LNK_EUNSUPPORTED;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_q_heads % d->num_kv_heads != 0) return LNK_EINVAL;
  const int g = d->num_q_heads / d->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return LNK_EUNSUPPORTED;
  if (d->num_pages <= 0 || d->num_rows <= 0 || d->pages_per_row <= 0) return LNK_EINVAL;
  if (d->window < 0 || !(d->scale >= 0.f)) return LNK_EINVAL;
  if (d->kv_dtype != LNK_KV_BF16 && d->kv_dtype != LNK_KV_E4M3) return LNK_EUNSUPPORTED;
  if (d->kv_dtype == LNK_KV_E4M3 && !(d->k_scale > 0.f && d->k_scale <= FLT_MAX && d->v_scale > 0.f &&
                                       d->v_scale <= FLT_MAX))
    return LNK_EINVAL;
  // TMA row coordinates and 32-bit position arithmetic must not overflow
  if (static_cast<long long>(d->num_kv_heads) * d->num_pages * kPage >= (1ll << 31)) return LNK_ERANGE;
  if (static_cast<long long>(d->pages_per_row) * kPage >= (1ll << 31)) return LNK_ERANGE;
  if (static_cast<long long>(d->num_rows) * d->pages_per_row >= (1ll << 31)) return LNK_ERANGE;
  return LNK_OK;
}

// Softmax scale in log2 units; for 8-bit pools the scores are computed on
// codes, so the key scale joins it.
float scale_log2(const lnk_attn_desc* d) {
  double s = d->scale > 0.f ? static_cast<double>(d->scale) : 1.0 / std::sqrt(static_cast<double>(d->head_dim));
  if (d->kv_dtype == LNK_KV_E4M3) s *= static_cast<double>(d->k_scale);
  return static_cast<float>(s * 1.4426950408889634);  // log2(e)
}

}  // namespace

cudaError_t set_max_dynamic_smem(const void* func, int bytes) {
  // cudaFuncSetAttribute only when a launch needs more than what was set on this device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[{func, dev}];
  if (have >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) have = bytes;
  return err;
}

cudaError_t prefer_max_shared(const void* func) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({func, dev})) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (err == cudaSuccess) done.insert({func, dev});
  return err;
}

cudaError_t occupancy_blocks(int* blocks, const void* func, int threads, size_t bytes) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, size_t>, int> done;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({func, dev, threads, bytes});
    if (it != done.end()) {
      *blocks = it->second;
      return cudaSuccess;
    }
  }
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, func, threads, bytes);
  if (err == cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    done[{func, dev, threads, bytes}] = *blocks;
  }
  return err;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::call_once(g_sm_once[dev], [dev] {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = n;
  });
  return g_sm_count[dev];
}

// Frequency table of lnk_rope_desc (float32 operations as the pages write them).
static lnk_status inv_freq_table(const lnk_rope_desc* rope, int head_dim, float* out) {
  if (rope == nullptr || out == nullptr || head_dim <= 0 || head_dim % 2 || head_dim > 128) return LNK_EINVAL;
  if (!(rope->theta > 1.0)) return LNK_EINVAL;
  const float theta32 = static_cast<float>(rope->theta);
  const float log_theta = static_cast<float>(std::log(static_cast<double>(theta32)));
  const float d32 = static_cast<float>(head_dim);
  for (int i = 0; i < head_dim / 2; ++i) {
    volatile float t = static_cast<float>(i) * 2.0f;  // volatile: keep each float32 rounding
    volatile float u = t / d32;
    volatile float e = (-u) * log_theta;
    out[i] = static_cast<float>(std::exp(static_cast<double>(e)));
  }
  if (rope->llama3) {
    const double factor = rope->factor, low = rope->low_freq_factor, high = rope->high_freq_factor;
    const double orig = rope->original_max_position;
    if (!(factor > 0.0) || !(high > low) || !(orig > 0.0)) return LNK_EINVAL;
    const double two_pi = 2.0 * 3.14159265358979323846;
    for (int i = 0; i < head_dim / 2; ++i) {
      const double inv = static_cast<double>(out[i]);
      const double wavelen = two_pi / inv;
      double v;
      if (wavelen > orig / low) {
        v = inv / factor;
      } else if (wavelen < orig / high) {
        v = inv;
      } else {
        const double smooth = (orig / wavelen - low) / (high - low);
        volatile double a = (1.0 - smooth) * (inv / factor);
        volatile double b = smooth * inv;
        v = a + b;
      }
      out[i] = static_cast<float>(v);
    }
  }
  return LNK_OK;
}

}  // namespace lnk

using namespace lnk;

extern "C" {

const char* lnk_status_string(lnk_status s) {
  switch (s) {
    case LNK_OK: return "LNK_OK";
    case LNK_EINVAL: return "LNK_EINVAL: invalid argument";
    case LNK_ERANGE: return "LNK_ERANGE: size out of range";
    case LNK_ECUDA: return "LNK_ECUDA: CUDA runtime error";
    case LNK_EUNSUPPORTED: return "LNK_EUNSUPPORTED: unsupported shape";
    case LNK_EWORKSPACE: return "LNK_EWORKSPACE: workspace missing or too small";
    case LNK_ENOSPACE: return "LNK_ENOSPACE: not enough free pages";
  }
  return "unknown lnk_status";
}

lnk_status lnk_rope_inv_freq(const lnk_rope_desc* rope, int32_t head_dim, float* out) {
  return inv_freq_table(rope, head_dim, out);
}

size_t lnk_paged_workspace_size(const lnk_attn_desc* desc, int32_t max_rows) {
  if (check_desc(desc) != LNK_OK || max_rows < 0 || max_rows > kMaxDecodeRows) return 0;
  // the largest grid a call can use (two CTAs per SM)
  const int grid = device_sm_count() * 2;
  if (grid <= 0) return 0;
  return decode_workspace_layout(max_rows, desc->num_kv_heads, desc->num_q_heads / desc->num_kv_heads,
                                 desc->head_dim, grid)
      .total;
}

}  // extern "C"

namespace lnk {

// Checks the append's arguments and fills its kernel parameters (shared by
// lnk_paged_append_rope and the fused decode step).  T > 0.
static lnk_status append_params(const lnk_attn_desc* desc, const lnk_rope_desc* rope, const lnk_bf16* q,
                                const lnk_bf16* k, const lnk_bf16* v, const int32_t* positions, const int32_t* rows,
                                const int32_t* slots, const int32_t* table, const lnk_bf16* q_norm_w,
                                const lnk_bf16* k_norm_w, float norm_eps, lnk_bf16* k_pool, lnk_bf16* v_pool,
                                lnk_bf16* q_out, int32_t T, int32_t* dev_status, AppendParams* out) {
  if (!q || !k || !v || !positions || !k_pool || !v_pool || !q_out) return LNK_EINVAL;
  if (slots == nullptr && table == nullptr) return LNK_EINVAL;
  if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 16) || !aligned(q_out, 4) || !aligned(k_pool, 16) ||
      !aligned(v_pool, 16) || (q_norm_w && !aligned(q_norm_w, 4)) || (k_norm_w && !aligned(k_norm_w, 4)))
    return LNK_EINVAL;
  if ((q_norm_w || k_norm_w) && !(norm_eps >= 0.f)) return LNK_EINVAL;
  if (rows == nullptr && slots == nullptr && T > desc->num_rows) return LNK_EINVAL;
  AppendParams& p = *out;
  std::memset(&p, 0, sizeof(p));
  {
    // the table is the same step after step: keep the last one per thread
    struct Cached {
      bool valid = false;
      int head_dim = 0;
      lnk_rope_desc rope;
      float table[64];
    };
    thread_local Cached c;
    const bool hit = c.valid && c.head_dim == desc->head_dim && rope != nullptr && c.rope.theta == rope->theta &&
                     c.rope.llama3 == rope->llama3 &&
                     (!rope->llama3 || (c.rope.factor == rope->factor && c.rope.low_freq_factor == rope->low_freq_factor &&
                                        c.rope.high_freq_factor == rope->high_freq_factor &&
                                        c.rope.original_max_position == rope->original_max_position));
    if (!hit) {
      const lnk_status st = inv_freq_table(rope, desc->head_dim, c.table);
      if (st != LNK_OK) {
        c.valid = false;
        return st;
      }
      c.valid = true;
      c.head_dim = desc->head_dim;
      c.rope = *rope;
    }
    std::memcpy(p.inv_freq, c.table, sizeof(float) * (desc->head_dim / 2));
  }
  p.q = q;
  p.k = k;
  p.v = v;
  p.positions = positions;
  p.rows = rows;
  p.slots = slots;
  p.table = table;
  p.q_norm_w = q_norm_w;
  p.k_norm_w = k_norm_w;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.q_out = q_out;
  p.status = dev_status;
  p.norm_eps = static_cast<double>(norm_eps);
  p.T = T;
  p.hq = desc->num_q_heads;
  p.hkv = desc->num_kv_heads;
  p.num_pages = desc->num_pages;
  p.num_rows = desc->num_rows;
  p.pages_per_row = desc->pages_per_row;
  p.kv8 = desc->kv_dtype == LNK_KV_E4M3;
  p.k_scale = desc->k_scale;
  p.v_scale = desc->v_scale;
  p.splits = 1;
  return LNK_OK;
}

}  // namespace lnk

extern "C" {

lnk_status lnk_paged_append_rope(const lnk_attn_desc* desc, const lnk_rope_desc* rope, const lnk_bf16* q,
                                 const lnk_bf16* k, const lnk_bf16* v, const int32_t* positions,
                                 const int32_t* rows, const int32_t* slots, const int32_t* table,
                                 const lnk_bf16* q_norm_w, const lnk_bf16* k_norm_w, float norm_eps,
                                 lnk_bf16* k_pool, lnk_bf16* v_pool, lnk_bf16* q_out, int32_t T,
                                 int32_t* dev_status, lnk_stream stream) {
  lnk_status st = check_desc(desc);
  if (st != LNK_OK) return st;
  if (T < 0) return LNK_EINVAL;
  if (T == 0) return LNK_OK;
  AppendParams p;
  st = append_params(desc, rope, q, k, v, positions, rows, slots, table, q_norm_w, k_norm_w, norm_eps, k_pool,
                     v_pool, q_out, T, dev_status, &p);
  if (st != LNK_OK) return st;
  return launch_append(p, desc->head_dim, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? LNK_OK
                                                                                                : LNK_ECUDA;
}

// The pools reach the kernel through their tensor maps (kmap, vmap).
// clear_counters: zero the workspace's counters on the stream right before the
// launch (after every check has passed), for a workspace whose previous
// contents are unknown.
// fuse: the fused decode step's append parameters (null: attention only).
static lnk_status decode_common(const lnk_attn_desc* desc, const lnk_bf16* q, const int32_t* positions,
                                const int32_t* table, lnk_bf16* out, int32_t B, void* workspace, size_t ws_bytes,
                                int32_t* dev_status, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t stream, bool clear_counters = false,
                                const AppendParams* fuse = nullptr) {
  if (B == 0) return LNK_OK;
  DecodeLaunch launch;
  const bool kv8 = desc->kv_dtype == LNK_KV_E4M3;
  if (decode_prepare(desc->head_dim, kv8, B, desc->num_kv_heads, &launch, fuse != nullptr) != cudaSuccess ||
      launch.grid <= 0)
    return LNK_ECUDA;
  const int group = desc->num_q_heads / desc->num_kv_heads;
  const DecodeWorkspace w = decode_workspace_layout(B, desc->num_kv_heads, group, desc->head_dim, launch.grid);
  if (workspace == nullptr || ws_bytes < w.total || !aligned(workspace, 256)) return LNK_EWORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p;
  p.q = q;
  p.positions = positions;
  p.table = table;
  p.out = out;
  p.status = dev_status;
  p.ws_next = reinterpret_cast<int32_t*>(ws + w.next);
  p.ws_count = reinterpret_cast<int32_t*>(ws + w.count);
  p.ws_ml = reinterpret_cast<float*>(ws + w.ml);
  p.ws_o = reinterpret_cast<float*>(ws + w.o);
  p.B = B;
  p.hq = desc->num_q_heads;
  p.hkv = desc->num_kv_heads;
  p.group = group;
  p.num_pages = desc->num_pages;
  p.pages_per_row = desc->pages_per_row;
  p.window = desc->window;
  p.scale_log2 = scale_log2(desc);
  p.out_scale = kv8 ? desc->v_scale : 1.f;
  std::memset(&p.ap, 0, sizeof(p.ap));
  p.fuse = 0;
  if (fuse != nullptr) {
    p.fuse = 1;
    p.ap = *fuse;
  }
  if (clear_counters && cudaMemsetAsync(ws, 0, w.ml, stream) != cudaSuccess) return LNK_ECUDA;
  return launch_decode(kmap, vmap, p, desc->head_dim, launch, stream) == cudaSuccess ? LNK_OK : LNK_ECUDA;
}

}  // extern "C"

namespace lnk {

lnk_status decode_entry(const lnk_attn_desc* desc, const lnk_bf16* q_roped, const int32_t* positions,
                        const int32_t* table, const lnk_bf16* k_pool, const lnk_bf16* v_pool, lnk_bf16* out,
                        int32_t B, void* workspace, size_t ws_bytes, int32_t* dev_status, lnk_stream stream,
                        bool clear_counters) {
  lnk_status st = check_desc(desc);
  if (st != LNK_OK) return st;
  if (B < 0 || B > desc->num_rows) return LNK_EINVAL;
  if (B > kMaxDecodeRows) return LNK_ERANGE;
  if (B == 0) return LNK_OK;
  if (!q_roped || !positions || !table || !k_pool || !v_pool || !out) return LNK_EINVAL;
  if (!aligned(q_roped, 16) || !aligned(out, 8) || !aligned(k_pool, 16) || !aligned(v_pool, 16)) return LNK_EINVAL;
  CUtensorMap kmap, vmap;
  if (!pool_map(&kmap, k_pool, *desc) || !pool_map(&vmap, v_pool, *desc)) return LNK_ECUDA;
  return decode_common(desc, q_roped, positions, table, out, B, workspace, ws_bytes, dev_status, kmap, vmap,
                       reinterpret_cast<cudaStream_t>(stream), clear_counters);
}

}  // namespace lnk

extern "C" {

lnk_status lnk_paged_decode_attn(const lnk_attn_desc* desc, const lnk_bf16* q_roped, const int32_t* positions,
                                 const int32_t* table, const lnk_bf16* k_pool, const lnk_bf16* v_pool,
                                 lnk_bf16* out, int32_t B, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                 lnk_stream stream) {
  return decode_entry(desc, q_roped, positions, table, k_pool, v_pool, out, B, workspace, ws_bytes, dev_status,
                      stream, false);
}

// The decode step is one kernel when every (row, kv head) pair can be one
// CTA's only work and the pairs occupy at least half the SMs, with at most
// kFuseMaxPages pages a pair (so that one long pair cannot hold up the launch
// for long).
static bool decode_step_fuses(const lnk_attn_desc* desc, int32_t B, int grid) {
  const long long pairs = static_cast<long long>(B) * desc->num_kv_heads;
  long long pair_pages = desc->pages_per_row;
  if (desc->window > 0) pair_pages = std::min<long long>(pair_pages, (desc->window - 1) / kPage + 2);
  return pairs <= grid && 2 * pairs >= device_sm_count() && pair_pages <= kFuseMaxPages;
}

int32_t lnk_paged_decode_step_launches(const lnk_attn_desc* desc, int32_t B) {
  if (check_desc(desc) != LNK_OK || B < 0 || B > desc->num_rows || B > kMaxDecodeRows) return -1;
  if (B == 0) return 0;
  DecodeLaunch launch;
  if (decode_prepare(desc->head_dim, desc->kv_dtype == LNK_KV_E4M3, B, desc->num_kv_heads, &launch, true) !=
          cudaSuccess ||
      launch.grid <= 0)
    return -1;
  return decode_step_fuses(desc, B, launch.grid) ? 1 : 2;
}

lnk_status lnk_paged_decode_step(const lnk_attn_desc* desc, const lnk_rope_desc* rope, const lnk_bf16* q,
                                 const lnk_bf16* k, const lnk_bf16* v, const int32_t* positions,
                                 const int32_t* table, const lnk_bf16* q_norm_w, const lnk_bf16* k_norm_w,
                                 float norm_eps, lnk_bf16* k_pool, lnk_bf16* v_pool, lnk_bf16* q_out,
                                 lnk_bf16* out, int32_t B, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                 lnk_stream stream) {
  lnk_status st = check_desc(desc);
  if (st != LNK_OK) return st;
  if (B < 0 || B > desc->num_rows) return LNK_EINVAL;
  if (B > kMaxDecodeRows) return LNK_ERANGE;
  if (B == 0) return LNK_OK;
  if (!table || !out || !aligned(q_out, 16) || !aligned(out, 8)) return LNK_EINVAL;
  AppendParams ap;
  st = append_params(desc, rope, q, k, v, positions, nullptr, nullptr, table, q_norm_w, k_norm_w, norm_eps, k_pool,
                     v_pool, q_out, B, dev_status, &ap);
  if (st != LNK_OK) return st;
  CUtensorMap kmap, vmap;
  if (!pool_map(&kmap, k_pool, *desc) || !pool_map(&vmap, v_pool, *desc)) return LNK_ECUDA;
  // the launch of the one-kernel form, and the attention kernel's launch of
  // the two-kernel form
  DecodeLaunch fused_launch, launch;
  const bool kv8 = desc->kv_dtype == LNK_KV_E4M3;
  if (decode_prepare(desc->head_dim, kv8, B, desc->num_kv_heads, &fused_launch, true) != cudaSuccess ||
      fused_launch.grid <= 0 ||
      decode_prepare(desc->head_dim, kv8, B, desc->num_kv_heads, &launch) != cudaSuccess || launch.grid <= 0)
    return LNK_ECUDA;
  const int group = desc->num_q_heads / desc->num_kv_heads;
  const bool fuses = decode_step_fuses(desc, B, fused_launch.grid);
  const DecodeWorkspace w = decode_workspace_layout(B, desc->num_kv_heads, group, desc->head_dim,
                                                    fuses ? fused_launch.grid : launch.grid);
  if (workspace == nullptr || ws_bytes < w.total || !aligned(workspace, 256)) return LNK_EWORKSPACE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fuses)
    return decode_common(desc, q_out, positions, table, out, B, workspace, ws_bytes, dev_status, kmap, vmap, s,
                         false, &ap);
  // otherwise the append, then attention
  if (launch_append(ap, desc->head_dim, s) != cudaSuccess) return LNK_ECUDA;
  return decode_common(desc, q_out, positions, table, out, B, workspace, ws_bytes, dev_status, kmap, vmap, s);
}

lnk_status lnk_paged_step_attn(const lnk_attn_desc* desc, const lnk_bf16* q_roped, const int32_t* rows,
                               const int32_t* positions, const int32_t* segments, const int32_t* step_positions,
                               const int32_t* table, const lnk_bf16* k_pool, const lnk_bf16* v_pool,
                               lnk_bf16* out, const int32_t* last, lnk_bf16* last_out, int32_t P, int32_t B,
                               int32_t M, void* workspace, size_t ws_bytes, int32_t* dev_status,
                               lnk_stream stream) {
  lnk_status st = check_desc(desc);
  if (st != LNK_OK) return st;
  if (P < 0 || B < 0 || M < 0 || B > desc->num_rows) return LNK_EINVAL;
  if (B > kMaxDecodeRows) return LNK_ERANGE;
  if (P == 0 && B == 0) return LNK_OK;
  if (!q_roped || !table || !k_pool || !v_pool || !out) return LNK_EINVAL;
  if (P > 0 && (!rows || !positions)) return LNK_EINVAL;
  if (B > 0 && !step_positions) return LNK_EINVAL;
  if (M > 0 && (!last || !last_out)) return LNK_EINVAL;
  if (P > 0 && desc->kv_dtype != LNK_KV_BF16) return LNK_EUNSUPPORTED;  // chunk kernel reads bf16 pools
  if (!aligned(q_roped, 16) || !aligned(out, 8) || !aligned(k_pool, 16) || !aligned(v_pool, 16)) return LNK_EINVAL;
  if (B > 0) {
    const size_t need = lnk_paged_workspace_size(desc, B);
    if (workspace == nullptr || need == 0 || ws_bytes < need) return LNK_EWORKSPACE;
  }
  CUtensorMap kmap, vmap;
  if (!pool_map(&kmap, k_pool, *desc) || !pool_map(&vmap, v_pool, *desc)) return LNK_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int group = desc->num_q_heads / desc->num_kv_heads;
  const size_t row_elems = static_cast<size_t>(desc->num_q_heads) * desc->head_dim;
  if (P > 0) {
    ChunkParams c;
    c.q = q_roped;
    c.rows = rows;
    c.positions = positions;
    c.segments = segments;
    c.table = table;
    c.out = out;
    c.status = dev_status;
    c.P = P;
    c.hq = desc->num_q_heads;
    c.hkv = desc->num_kv_heads;
    c.group = group;
    c.num_pages = desc->num_pages;
    c.num_rows = desc->num_rows;
    c.pages_per_row = desc->pages_per_row;
    c.window = desc->window;
    c.tile_tokens = 128 / group;
    c.num_tiles = (P + kChunkHalves * c.tile_tokens - 1) / (kChunkHalves * c.tile_tokens);
    c.scale_log2 = scale_log2(desc);
    if (launch_chunk(kmap, vmap, c, desc->head_dim, s) != cudaSuccess) return LNK_ECUDA;
  }
  if (B > 0) {
    st = decode_common(desc, q_roped + static_cast<size_t>(P) * row_elems, step_positions, table,
                       out + static_cast<size_t>(P) * row_elems, B, workspace, ws_bytes, dev_status, kmap, vmap, s);
    if (st != LNK_OK) return st;
  }
  if (M > 0) {
    if (launch_gather_last(out, last, last_out, M, P, static_cast<int>(row_elems), dev_status, s) != cudaSuccess)
      return LNK_ECUDA;
  }
  return LNK_OK;
}

}  // extern "C"
