// K2 + K3: paged split-KV decode attention with a fused log-sum-exp combine.
//
// Work decomposition.  Decode row b at position p sees keys
// [max(0, p - window + 1), p], i.e. np_b pages of 64 (the first and last may
// be partial).  Each (row, kv head) pair is a run of np_b page-heads; the runs
// of all pairs, (b, h) with h fastest, are laid end to end and the resulting
// stream of page-heads is cut into equal chunks: one per persistent CTA, or
// kChunksPerCta per CTA when the launch has many (row, kv head) pairs (at
// least 5 per CTA).  CTA c starts with chunk c and then claims further chunks
// from a counter in the workspace, so that CTAs whose pages arrive slower
// take fewer chunks (the last claimant returns the counter to zero).  The
// part of a pair inside one chunk is a segment.  A pair that falls inside one
// chunk is finished there (output written directly).  A pair cut by chunk
// boundaries leaves one partial result per chunk (unnormalised output,
// running max, running sum; pair q in chunk i writes segment q + i, unique
// because consecutive pairs never go back to an earlier chunk); each such
// chunk then increments the pair's counter, and the last one to arrive merges
// the partials and writes the output (the counter returns to zero).  Within a
// chunk, the segment it shares with the next chunk is processed first, so
// that cut pairs finish early instead of in the tail.
//
// CTA structure (192 threads, warp-specialised):
//  * warp 4, producer: one lane walks the CTA's page-heads, reads the page
//    table, and loads each page's K and V (64 positions x head_dim bf16,
//    contiguous in the head-major pool) with 2-D TMA tile copies into a ring
//    of shared-memory stages (128-byte swizzle), plus the segment's G query
//    rows (one 1-D bulk copy) on a segment's first page; all complete on the
//    stage's "full" mbarrier.
//  * warps 0-3, consumers: warp w owns keys 16w .. 16w + 15 of every page.
//    It copies its K and V fragments to registers (ldmatrix), releases the
//    stage at once, and then computes
//      S^T[16 keys, 8 heads] = K[16 keys, D] Q^T   (mma m16n8k16, keys as M,
//                                                   the GQA group padded to N)
//      O^T[D, 8 heads]      += V^T[D, 16 keys] P^T (P^T via movmatrix.trans
//                                                   of the S fragment)
//    with an online softmax in the log2 domain.  At a segment's end each warp
//    hands its state to the epilogue through one of two staging slots.
//  * warp 5, epilogue: merges the four warps' states of each segment and
//    writes the output (whole pairs) or the partial, counter and, for the
//    last arriver, the merged output of a cut pair.  Consumers never wait on
//    global memory.
// 8-bit pools (E4M3 codes, one byte per element): a page of one head is one
// 128-byte-wide TMA box (the codes viewed as 16-bit pairs), so a stage holds
// half the bytes and two CTAs share an SM (twice the consumer warps for the
// same bytes in flight).  The consumers convert codes
// to f16 (exact) and use the f16 mma.  No byte transposes are needed:
//  * K: ldmatrix of the 16-bit view gives a lane 4 consecutive dimensions of
//    one key; read as k = (4c, 4c+1 | 4c+2, 4c+3) of a 16-dimension step,
//    with the query fragment read in the same order;
//  * V: a lane loads 4-byte words of keys c, c+4, c+8, c+12 and pairs their
//    bytes (prmt), so the 16 keys of a step appear in the order
//    m -> (m & 8) | ((m >> 1) & 3) | ((m & 1) << 2); Q.K takes its key rows
//    in that same order, so P^T from movmatrix matches; the 4 dimensions a
//    lane holds make the M rows of two d-tiles, undone when O is staged.
// The key scale multiplies the softmax scale, the value scale the output.
// The per-row prologue (visible pages, prefix sums, the producer's plan of its
// first chunk) reads only positions and the table, so it overlaps the
// previous kernel on the stream (programmatic dependent launch); the kernel
// waits for that kernel before touching q or the pool.  The producer warp
// waits last, right before its first copy, once its first stage's record is
// written; with one short pair per CTA it also asks L2 to prefetch the pair's
// pages before the wait (a prefetch reads nothing into the kernel).  The
// kernel lets the next kernel on the stream start early in the same way.
//
// Sources: "Phi-3 Mini 4K Instruct -- files", src/attention.linnet
// (decode_rows: a row attends over itself up to its position; window_mask;
// scale rsqrt(head_dim)); "Mistral 7B Instruct v0.3", Entries table
// (decode_paged: the pool, pages of 64, table[b]).
#include "common.cuh"
#include "ptx.cuh"
#include "rope_math.cuh"

namespace lnk {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kEpilogueWarp = 5;
constexpr int kThreads = 6 * 32;
#ifndef LNK_DECODE_STAGES
#define LNK_DECODE_STAGES 4
#endif
constexpr int kStages = LNK_DECODE_STAGES;  // K+V pages in flight per CTA (bf16 pools)
constexpr int kSegFirst = 1;
constexpr int kSegLast = 2;
constexpr int kPairWhole = 4;
constexpr int kEnd = 8;   // no more work: passed from the producer to the consumers and the epilogue

struct StageInfo {
  int b, h, klo, khi, flags, seg, nseg, c0;
};

// Kernel variants: bf16 pools with one CTA per SM (4 stages), bf16 pools
// with two CTAs per SM (2 stages each, for launches with many (row, kv head)
// pairs), 8-bit pools with two CTAs per SM (4 stages of half the bytes).
constexpr int kModeBf16 = 0, kModeBf16Two = 1, kModeE4m3 = 2;

template <int D, int MODE>
struct DecodeSmem {
  static constexpr bool F8 = MODE == kModeE4m3;
  static constexpr int NB = F8 ? 1 : boxes_for(D);         // TMA boxes per page of one head
  static constexpr int kStages = MODE == kModeBf16Two ? 2 : lnk::kStages;
  static constexpr int kStageBytes = 2 * NB * kBoxBytes;  // K boxes, then V boxes
  static constexpr int kQBytes = kMaxGroup * D * 2;       // query rows of the stage's segment
  static constexpr int kOStride = D + 4;                  // padded staging row
  static constexpr int kSlotFloats = kConsumerWarps * kMaxGroup * kOStride;
  static constexpr size_t stages = 0;
  static constexpr size_t qbuf = stages + size_t(kStages) * kStageBytes;
  static constexpr size_t bars = qbuf + size_t(kStages) * kQBytes;
  // full[kStages], empty[kStages], slot_full[2], slot_empty[2], appended
  // (rounded up to 16 bytes: the staging slots after them are read as float4)
  static constexpr size_t info = bars + ((2 * kStages + 5) * sizeof(uint64_t) + 15) / 16 * 16;
  static constexpr size_t slot_info = info + kStages * sizeof(StageInfo);
  static constexpr size_t ostage = slot_info + 2 * sizeof(StageInfo);
  static constexpr size_t mstage = ostage + 2 * size_t(kSlotFloats) * 4;
  static constexpr size_t lstage = mstage + 2 * kConsumerWarps * kMaxGroup * 4;
  static constexpr size_t epi = lstage + 2 * kConsumerWarps * kMaxGroup * 4;   // epilogue scratch
  static constexpr size_t misc = epi + 2 * kMaxGroup * 4;                       // abort flag, scan sums
  static constexpr size_t pref = misc + 64;
  // Fused decode step: the rotation coefficients [2 kinds][D / 2] live in the
  // epilogue's staging slots, which nothing writes before the pair's last page
  // has landed (that page waits for the append, the append's last reader of
  // the coefficients).
  static constexpr size_t coef = ostage;
  static_assert(2 * (D / 2) * sizeof(rope::Coefs) <= 2 * size_t(kSlotFloats) * 4, "coefficients fit the staging slots");
  static_assert(ostage % 16 == 0 && kOStride % 4 == 0, "staging rows are read as float4");
  static size_t bytes(int B) { return pref + size_t(B + 1) * 4 + 1024; }  // + alignment slack
};

__device__ __forceinline__ int visible_pages(int pos, int window, int pages_per_row, int* bad) {
  if (pos < 0) return 0;
  if (pos >= pages_per_row * kPage) {
    *bad = LNK_DEV_BAD_POSITION;
    return 0;
  }
  const int lo = window > 0 ? max(0, pos - window + 1) : 0;
  return pos / kPage - lo / kPage + 1;
}

// Where page-head `gi` of the flattened stream lies, and the per-pair values
// the producer needs (computed once per pair, not per page).
struct Cursor {
  int b, h, j, np, pos, lo, first_page;
  int seg, c0, nseg, whole;
  const int* trow;
};

__device__ __forceinline__ void locate(Cursor& c, long long gi, const int* pref, const DecodeParams& p,
                                       long long start, long long end, long long per, long long chunk) {
  int lo_b = 0, hi_b = p.B - 1;  // largest b with hkv * pref[b] <= gi
  while (lo_b < hi_b) {
    const int mid = (lo_b + hi_b + 1) >> 1;
    if (static_cast<long long>(pref[mid]) * p.hkv <= gi) lo_b = mid; else hi_b = mid - 1;
  }
  c.b = lo_b;
  c.np = pref[c.b + 1] - pref[c.b];
  const long long rem = gi - static_cast<long long>(pref[c.b]) * p.hkv;
  c.h = static_cast<int>(rem / c.np);
  c.j = static_cast<int>(rem % c.np);
  c.pos = p.positions[c.b];
  c.lo = p.window > 0 ? max(0, c.pos - p.window + 1) : 0;
  c.first_page = c.lo / kPage;
  c.trow = p.table + static_cast<long long>(c.b) * p.pages_per_row;
  const long long pair_start = gi - c.j;
  const long long pair_end = pair_start + c.np;
  c.whole = pair_start >= start && pair_end <= end;
  c.c0 = static_cast<int>(pair_start / per);
  c.nseg = static_cast<int>((pair_end - 1) / per) - c.c0 + 1;
  c.seg = c.b * p.hkv + c.h + static_cast<int>(chunk);
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == kModeBf16 ? 1 : 2)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  using L = DecodeSmem<D, MODE>;
  constexpr bool F8 = L::F8;
  constexpr int NB = L::NB;
  constexpr int kStages = L::kStages;
  constexpr int DK = D / 16;  // k-steps of Q.K and d-tiles of P.V
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* slot_full = empty_bar + kStages;  // [2]: consumer warps -> epilogue
  uint64_t* slot_empty = slot_full + 2;       // [2]: epilogue -> consumer warps
  uint64_t* appended = slot_empty + 2;        // fused step: the pair's new K/V row is in the pool
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + L::info);
  StageInfo* slot_info = reinterpret_cast<StageInfo*>(smem + L::slot_info);
  float* ost = reinterpret_cast<float*>(smem + L::ostage);
  float* mst = reinterpret_cast<float*>(smem + L::mstage);
  float* lst = reinterpret_cast<float*>(smem + L::lstage);
  int* misc = reinterpret_cast<int*>(smem + L::misc);  // [0] abort, [2..7] warp sums of the scan, [8] longest pair
  volatile int* abort_flag = misc;
  int* pref = reinterpret_cast<int*>(smem + L::pref);

  // Let the next kernel on the stream start its own prologue while this one
  // runs; it must wait for this grid (griddepcontrol.wait) before it reads
  // the output or writes anything this kernel reads.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int B = p.B;
  const int G = p.group;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(full_bar + s), 1);
      mbar_init(smem_addr(empty_bar + s), kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(slot_full + i), kConsumerWarps);
      mbar_init(smem_addr(slot_empty + i), 1);
    }
    mbar_init(smem_addr(appended), 1);
    misc[0] = 0;
    misc[8] = 0;  // longest pair (pages)
    fence_mbarrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_descriptor(&kmap);
    tma_prefetch_descriptor(&vmap);
  }

  // ---- per-row visible page counts and their prefix sums (all threads) ----
  {
    const int chunk = (B + kThreads - 1) / kThreads;
    const int r0 = min(B, tid * chunk), r1 = min(B, r0 + chunk);
    int bad = 0, run = 0, longest = 0;
    for (int b = r0; b < r1; ++b) {
      const int np = visible_pages(p.positions[b], p.window, p.pages_per_row, &bad);
      longest = max(longest, np);
      run += np;
      pref[b + 1] = run;
    }
    if (bad && p.status != nullptr && blockIdx.x == 0) atomicOr(p.status, bad);
    int incl = run;  // inclusive scan of the per-thread totals across the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) misc[2 + warp] = incl;
    __syncthreads();  // (also orders misc[8] = 0 above before the maxima below)
    if (longest > 0) atomicMax(misc + 8, longest);
    int off = incl - run;
    for (int w = 0; w < warp; ++w) off += misc[2 + w];
    for (int b = r0; b < r1; ++b) pref[b + 1] += off;
    if (tid == 0) pref[0] = 0;
    __syncthreads();
  }

  const long long total = static_cast<long long>(pref[B]) * p.hkv;
  const long long pairs = static_cast<long long>(B) * p.hkv;
  // At most one pair per CTA, none longer than twice a CTA's share: each
  // chunk is one whole pair (no partial results, no merges).
  // (The fused step always takes one pair per CTA: the host calls it only when
  // the pairs fit the grid and are short.)
  const bool pair_chunks =
      p.fuse || (pairs <= gridDim.x && 2 * ((total + gridDim.x - 1) / gridDim.x) >= misc[8]);
  // Several chunks per CTA only when pairs are many (and so short) against a
  // CTA's share: each chunk boundary cuts a pair, and a cut pair costs a
  // partial result and a merge.
  // (8-bit pools keep one chunk per CTA: there, finer chunks measured slower,
  // their cut pairs' partials and merges costing more than the balance gained.)
  const int chunks_per_cta = !F8 && static_cast<long long>(B) * p.hkv >= 5ll * gridDim.x ? kChunksPerCta : 1;
  const long long per = (total + chunks_per_cta * gridDim.x - 1) / (chunks_per_cta * gridDim.x);  // chunk size
  const long long nchunks = pair_chunks ? pairs : (per > 0 ? (total + per - 1) / per : 0);
  // page-head range of a chunk
  auto chunk_range = [&](long long c, long long& s0, long long& s1) {
    if (pair_chunks) {
      const int b = static_cast<int>(c / p.hkv), h = static_cast<int>(c % p.hkv);
      const int np = pref[b + 1] - pref[b];
      s0 = static_cast<long long>(pref[b]) * p.hkv + static_cast<long long>(h) * np;
      s1 = s0 + np;
    } else {
      s0 = c * per;
      s1 = min(total, s0 + per);
    }
  };

  // The table entries of the cursor's page and of the pair's next three
  // pages (0 past the pair's last page), read together: the producer keeps
  // this window of entries, so that a page's TMA copies never wait for the
  // table once the window is full.
  auto window_entries = [&](const Cursor& c, int& e0, int& e1, int& e2, int& e3) {
    const int* t = c.trow + c.first_page + c.j;
    const int left = c.np - c.j;
    e0 = left > 0 ? t[0] : 0;
    e1 = left > 1 ? t[1] : 0;
    e2 = left > 2 ? t[2] : 0;
    e3 = left > 3 ? t[3] : 0;
  };
  // The producer's plan of a chunk: its page-head range, the order of its
  // segments (the one it shares with the next chunk first), the cursor at the
  // first page-head and the window of table entries there.
  struct ChunkPlan {
    long long start, end, rb0, re0, rb1, re1;  // ranges in order: [rb0, re0), then [rb1, re1)
    int nranges, e0, e1, e2, e3;
    Cursor cur;
  };
  auto plan_chunk = [&](long long chunk, ChunkPlan& pl) {
    chunk_range(chunk, pl.start, pl.end);
    pl.nranges = 0;
    if (pl.start >= pl.end) return;
    locate(pl.cur, pl.end - 1, pref, p, pl.start, pl.end, per, chunk);
    const long long last_seg = max(pl.start, pl.end - 1 - pl.cur.j);
    const bool last_cut = (pl.end - 1 - pl.cur.j) + pl.cur.np > pl.end;
    if (last_cut && last_seg > pl.start) {
      pl.rb0 = last_seg; pl.re0 = pl.end;
      pl.rb1 = pl.start; pl.re1 = last_seg;
      pl.nranges = 2;
    } else {
      pl.rb0 = pl.start; pl.re0 = pl.end;
      pl.rb1 = pl.re1 = pl.end;
      pl.nranges = 1;
    }
    locate(pl.cur, pl.rb0, pref, p, pl.start, pl.end, per, chunk);
    window_entries(pl.cur, pl.e0, pl.e1, pl.e2, pl.e3);
  };
  // Fused step, before the wait (positions and the table only): the sine and
  // cosine of row b's angles (threads below D / 2) and the pool slot of its
  // token (the epilogue warp's last lane) for this CTA's pair (b, h).
  constexpr int H = D / 2;
  const bool fused = p.fuse && static_cast<long long>(blockIdx.x) < pairs;
  const int f_row = fused ? static_cast<int>(blockIdx.x / p.hkv) : 0;
  const int f_head = fused ? static_cast<int>(blockIdx.x % p.hkv) : 0;
  const int fpos = fused ? p.positions[f_row] : -1;
  rope::DF f_sn{0.f, 0.f}, f_cs{0.f, 0.f};
  if (fused && tid < H && fpos >= 0) rope::angle_sincos(fpos, p.ap.inv_freq[tid], f_sn, f_cs);
  long long f_slot = -1;
  int f_bad = 0;
  if (fused && warp == kEpilogueWarp && lane == 31 && fpos >= 0) {
    if (fpos >= p.pages_per_row * kPage) {
      f_bad = LNK_DEV_BAD_POSITION;
    } else {
      const int page = p.table[static_cast<long long>(f_row) * p.pages_per_row + fpos / kPage];
      if (page < 0 || page >= p.num_pages) f_bad = LNK_DEV_BAD_PAGE;
      else f_slot = static_cast<long long>(page) * kPage + fpos % kPage;
    }
  }

  // The first chunk's plan reads only positions and the table, so the
  // producer makes it before the wait (neither may be written by the
  // previous kernel on the stream).
  ChunkPlan first_plan;
  first_plan.nranges = 0;
  if (warp == kProducerWarp && lane == 0 && static_cast<long long>(blockIdx.x) < nchunks) {
    plan_chunk(blockIdx.x, first_plan);
    // One short pair per CTA: through a short ring its pages would take a
    // DRAM round trip per ring's worth, so all of them are prefetched into L2
    // first.  (Prefetches only: whatever the previous kernel writes to these
    // pages still reaches L2 before this kernel's copies read them, after the
    // wait.)
    if (pair_chunks && first_plan.nranges > 0) {
      const Cursor& c = first_plan.cur;
      for (int j = c.j; j < c.np; ++j) {
        const int page = c.trow[c.first_page + j];
        if (page >= 0 && page < p.num_pages) {
          const int y = (c.h * p.num_pages + page) * kPage;
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            tma_prefetch_l2_2d(&kmap, nb * kBoxCols, y);
            tma_prefetch_l2_2d(&vmap, nb * kBoxCols, y);
          }
        }
      }
    }
  }

  // Wait for the previous kernel on the stream (it writes q and the pool).
  // The producer warp waits later, right before its first copy: the first
  // stage's bookkeeping then runs before the wait, which also brings the
  // producer's code into the instruction cache (run first after the wait, it
  // took about 1200 cycles to reach the first copy).
  if (warp != kProducerWarp) asm volatile("griddepcontrol.wait;" ::: "memory");

  // rows with nothing to attend to get a zero output (the producer warp does
  // not take part: it has not waited yet)
  if (warp != kProducerWarp) {
    const int zt = warp < kProducerWarp ? tid : tid - 32;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
      if (pref[b + 1] == pref[b]) {
        uint32_t* o = reinterpret_cast<uint32_t*>(p.out + static_cast<size_t>(b) * p.hq * D);
        for (int i = zt; i < p.hq * D / 2; i += kThreads - 32) o[i] = 0u;
      }
    }
  }
  if (static_cast<long long>(blockIdx.x) >= nchunks) return;

  // ---- fused step: the append's work for this CTA's pair (b, h) ----
  // Consumer warp w rotates query heads w, w + 4 of the pair into q_out and
  // into stage 0's query rows; the epilogue warp rotates the key head into
  // the pool slot and copies the value row there, then tells the producer,
  // which loads the pair's last page (the one holding the slot) only after
  // that.  The arithmetic is rope_math.cuh's, as in the append kernel.
  if (fused && warp != kProducerWarp) {
    rope::Coefs* s_coef = reinterpret_cast<rope::Coefs*>(smem + L::coef);  // [queries, keys][D / 2]
    const AppendParams& ap = p.ap;
    if (tid < H && fpos >= 0) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint16_t* w = which == 0 ? ap.q_norm_w : ap.k_norm_w;
        float g1 = 1.f, g2 = 1.f;
        if (w != nullptr) {
          g1 = __uint_as_float(static_cast<uint32_t>(w[tid]) << 16);
          g2 = __uint_as_float(static_cast<uint32_t>(w[tid + H]) << 16);
        }
        s_coef[which * H + tid] = rope::coefs_of(f_sn, f_cs, g1, g2);
      }
    }
    named_barrier_sync(1, (kConsumerWarps + 1) * 32);  // the consumer warps and the epilogue warp
    const bool has = lane < D / 4;  // lanes holding elements (e, e + 1) and (e + D/2, e + D/2 + 1)
    const int e = 2 * lane;
    const bool live = fpos >= 0;
    if (warp < kConsumerWarps) {
      uint16_t* sq = reinterpret_cast<uint16_t*>(smem + L::qbuf);  // stage 0's query rows [G][D]
      const bool normed = ap.q_norm_w != nullptr;
      for (int g = warp; g < G; g += kConsumerWarps) {
        const size_t row = (static_cast<size_t>(f_row) * p.hq + static_cast<size_t>(f_head) * G + g) * D;
        uint32_t xlo = 0u, xhi = 0u;
        if (has && live) {
          xlo = *reinterpret_cast<const uint32_t*>(ap.q + row + e);
          xhi = *reinterpret_cast<const uint32_t*>(ap.q + row + H + e);
        }
        rope::DF r{1.f, 0.f};
        if (normed && live) r = rope::rms_factor(rope::head_sumsq(xlo, xhi), D, ap.norm_eps);
        uint32_t lo = 0u, hi = 0u;  // (zero for an inactive row)
        if (has && live) rope::rotate_pairs(xlo, xhi, s_coef, e, normed, r, lo, hi);
        if (has) {
          *reinterpret_cast<uint32_t*>(ap.q_out + row + e) = lo;
          *reinterpret_cast<uint32_t*>(ap.q_out + row + H + e) = hi;
          *reinterpret_cast<uint32_t*>(sq + g * D + e) = lo;
          *reinterpret_cast<uint32_t*>(sq + g * D + H + e) = hi;
        }
      }
      named_barrier_sync(2, kConsumerWarps * 32);  // every query row is in shared memory
    } else {
      const long long slot = __shfl_sync(0xffffffffu, f_slot, 31);
      if (lane == 31 && f_bad && p.status != nullptr) atomicOr(p.status, f_bad);
      if (slot >= 0) {
        const size_t src = (static_cast<size_t>(f_row) * p.hkv + f_head) * D;
        const size_t dst = (static_cast<size_t>(f_head) * p.num_pages * kPage + static_cast<size_t>(slot)) * D;
        const bool normed = ap.k_norm_w != nullptr;
        // (the key and value rows are loaded together, before any store)
        uint32_t xlo = 0u, xhi = 0u;
        uint4 vx = make_uint4(0u, 0u, 0u, 0u);
        if (has) {
          xlo = *reinterpret_cast<const uint32_t*>(ap.k + src + e);
          xhi = *reinterpret_cast<const uint32_t*>(ap.k + src + H + e);
        }
        if (lane < D / 8) vx = reinterpret_cast<const uint4*>(ap.v + src)[lane];
        rope::DF r{1.f, 0.f};
        if (normed) r = rope::rms_factor(rope::head_sumsq(xlo, xhi), D, ap.norm_eps);
        if (has) {
          uint32_t lo, hi;
          rope::rotate_pairs(xlo, xhi, s_coef + H, e, normed, r, lo, hi);
          if (ap.kv8) {
            uint8_t* k8 = reinterpret_cast<uint8_t*>(ap.k_pool) + dst;
            *reinterpret_cast<uint16_t*>(k8 + e) = rope::e4m3_pair(lo, ap.k_scale);
            *reinterpret_cast<uint16_t*>(k8 + H + e) = rope::e4m3_pair(hi, ap.k_scale);
          } else {
            *reinterpret_cast<uint32_t*>(ap.k_pool + dst + e) = lo;
            *reinterpret_cast<uint32_t*>(ap.k_pool + dst + H + e) = hi;
          }
        }
        if (lane < D / 8) {
          const uint4 x = vx;
          if (ap.kv8) {
            uint2 codes;
            codes.x = rope::e4m3_pair(x.x, ap.v_scale) | (static_cast<uint32_t>(rope::e4m3_pair(x.y, ap.v_scale)) << 16);
            codes.y = rope::e4m3_pair(x.z, ap.v_scale) | (static_cast<uint32_t>(rope::e4m3_pair(x.w, ap.v_scale)) << 16);
            reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(ap.v_pool) + dst)[lane] = codes;
          } else {
            reinterpret_cast<uint4*>(ap.v_pool + dst)[lane] = x;
          }
        }
        // the producer's tensor copies (async proxy) read these rows next
        fence_proxy_async_global();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(appended));
    }
  }

  if (warp == kProducerWarp) {
    // ============================== producer ==============================
    if (lane != 0) return;
    // (fused step: the consumers write the rotated queries themselves)
    const uint32_t q_bytes = fused ? 0u : static_cast<uint32_t>(G * D * 2);
    int k = 0;
    bool stop = false, waited = false;
    Cursor cur;
    for (long long chunk = blockIdx.x; chunk < nchunks && !stop;) {
      ChunkPlan pl;
      if (chunk == blockIdx.x) pl = first_plan; else plan_chunk(chunk, pl);
      const long long start = pl.start, end = pl.end;
      for (int rg = 0; rg < pl.nranges && !stop; ++rg) {
        const long long rb = rg == 0 ? pl.rb0 : pl.rb1, re = rg == 0 ? pl.re0 : pl.re1;
        int e0 = pl.e0, e1 = pl.e1, e2 = pl.e2, e3 = pl.e3;  // table window at the cursor
        if (rg == 0) {
          cur = pl.cur;
        } else {
          locate(cur, rb, pref, p, start, end, per, chunk);
          window_entries(cur, e0, e1, e2, e3);
        }
        for (long long gi = rb; gi < re; ++gi, ++k) {
          const int s = k % kStages;
          if (k >= kStages && !mbar_wait(smem_addr(empty_bar + s), ((k / kStages) - 1) & 1, abort_flag)) {
            stop = true;
            break;
          }
          // fused step: the pair's last page holds the new token, written by
          // the epilogue warp; load it only after that write
          if (fused && cur.j == cur.np - 1 && !mbar_wait(smem_addr(appended), 0, abort_flag)) {
            stop = true;
            break;
          }
          const int lp = cur.first_page + cur.j;
          const int page = e0;
          StageInfo si;
          si.b = cur.b;
          si.h = cur.h;
          si.klo = max(cur.lo - lp * kPage, 0);
          si.khi = min(cur.pos - lp * kPage + 1, kPage);
          const bool first = gi == rb || cur.j == 0;
          si.flags = (first ? kSegFirst : 0) | ((gi == re - 1 || cur.j == cur.np - 1) ? kSegLast : 0) |
                     (cur.whole ? kPairWhole : 0);
          si.seg = cur.seg;
          si.nseg = cur.nseg;
          si.c0 = cur.c0;
          const bool valid = page >= 0 && page < p.num_pages;
          if (!valid) {
            if (p.status != nullptr) atomicOr(p.status, LNK_DEV_BAD_PAGE);
            si.klo = si.khi = 0;
          }
          info[s] = si;
          const uint32_t fb = smem_addr(full_bar + s);
          const uint32_t tx = (valid ? static_cast<uint32_t>(L::kStageBytes) : 0u) + (first ? q_bytes : 0u);
          if (tx) mbar_arrive_expect_tx(fb, tx); else mbar_arrive(fb);
          if (!waited) {  // (the previous kernel writes q and the pool)
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
          }
          if (first && q_bytes > 0) {
            const uint16_t* qsrc = p.q + (static_cast<size_t>(cur.b) * p.hq + static_cast<size_t>(cur.h) * G) * D;
            bulk_load(smem_addr(smem + L::qbuf + size_t(s) * L::kQBytes), qsrc, q_bytes, fb);
          }
          if (valid) {
            const uint32_t kdst = smem_addr(smem + L::stages + size_t(s) * L::kStageBytes);
            const uint32_t vdst = kdst + NB * kBoxBytes;
            const int y = (cur.h * p.num_pages + page) * kPage;
  #pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              tma_load_2d(kdst + nb * kBoxBytes, &kmap, nb * kBoxCols, y, fb);
              tma_load_2d(vdst + nb * kBoxBytes, &vmap, nb * kBoxCols, y, fb);
            }
          }
          // advance to the next page-head (and the table window with it)
          if (++cur.j == cur.np && gi + 1 < re) {
            locate(cur, gi + 1, pref, p, start, end, per, chunk);
            window_entries(cur, e0, e1, e2, e3);
          } else {
            e0 = e1;
            e1 = e2;
            e2 = e3;
            e3 = cur.np - cur.j > 3 ? cur.trow[cur.first_page + cur.j + 3] : 0;
          }
        }
      }
      // the next chunk: claims are handed out in order, nchunks in all; the
      // last claimant returns the counter to zero for the next launch (with
      // no more chunks than CTAs there is nothing to claim)
      if (nchunks <= static_cast<long long>(gridDim.x)) break;
      const int v = atomicAdd(p.ws_next, 1);
      if (v == static_cast<int>(nchunks) - 1) atomicExch(p.ws_next, 0);
      chunk = static_cast<long long>(v) + gridDim.x;
    }
    // end of the work: one more stage, carrying no data
    {
      const int s = k % kStages;
      if (stop || (k >= kStages && !mbar_wait(smem_addr(empty_bar + s), ((k / kStages) - 1) & 1, abort_flag))) {
        // aborted: the consumers stop on the abort flag
      } else {
        StageInfo si{};
        si.flags = kEnd;
        info[s] = si;
        mbar_arrive(smem_addr(full_bar + s));
        ++k;
      }
    }
    // Drain: do not leave the CTA while a copy may still land in its memory.
    const int issued = k;
    for (int kk = max(0, issued - kStages); kk < issued; ++kk) {
      const uint32_t fb = smem_addr(full_bar + kk % kStages);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(fb, (kk / kStages) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {
      }
    }
    if (*abort_flag && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
    return;
  }

  if (warp == kEpilogueWarp) {
    // ============================== epilogue ==============================
    float* eml = reinterpret_cast<float*>(smem + L::epi);  // [2][kMaxGroup]: max, sum per head
    constexpr int D4 = D / 4;
    for (int n = 0;; ++n) {
      const int slot = n & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(slot_full + slot), (n >> 1) & 1, abort_flag))) break;
      const StageInfo si = slot_info[slot];
      if (si.flags & kEnd) break;
      const float* os = ost + size_t(slot) * L::kSlotFloats;
      const float* ms = mst + slot * kConsumerWarps * kMaxGroup;
      const float* ls = lst + slot * kConsumerWarps * kMaxGroup;
      const bool whole = (si.flags & kPairWhole) != 0;
      uint16_t* out_pair = p.out + (static_cast<size_t>(si.b) * p.hq + static_cast<size_t>(si.h) * G) * D;
      const int q = si.b * p.hkv + si.h;
      // per head: merged max and sum of the four warps
      if (lane < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, ms[w * kMaxGroup + lane]);
        float Ls = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = ms[w * kMaxGroup + lane];
            if (mw != -INFINITY) Ls += ls[w * kMaxGroup + lane] * exp2f(mw - M);
          }
        }
        eml[lane] = M;
        eml[kMaxGroup + lane] = Ls;
      }
      __syncwarp();
      for (int it = lane; it < G * D4; it += 32) {
        const int g = it / D4, d = (it % D4) * 4;
        const float M = eml[g], Ls = eml[kMaxGroup + g];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = ms[w * kMaxGroup + g];
            const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
            const float4 v = *reinterpret_cast<const float4*>(os + (w * kMaxGroup + g) * L::kOStride + d);
            acc.x += v.x * f;
            acc.y += v.y * f;
            acc.z += v.z * f;
            acc.w += v.w * f;
          }
        }
        if (whole) {
          const float inv = Ls > 0.f ? p.out_scale / Ls : 0.f;
          uint2 pk;
          pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
          *reinterpret_cast<uint2*>(out_pair + g * D + d) = pk;
        } else {
          *reinterpret_cast<float4*>(p.ws_o + (static_cast<size_t>(si.seg) * G + g) * D + d) = acc;
          if (d == 0) {
            p.ws_ml[(static_cast<size_t>(si.seg) * G + g) * 2 + 0] = M;
            p.ws_ml[(static_cast<size_t>(si.seg) * G + g) * 2 + 1] = Ls;
          }
        }
      }
      __syncwarp();
      // staging slot consumed
      if (lane == 0) mbar_arrive(smem_addr(slot_empty + slot));
      if (!whole) {
        // publish the partial, then count the pair's finished segments
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          const int old = atomicAdd(p.ws_count + q, 1);
          last = old == si.nseg - 1;
          if (last) p.ws_count[q] = 0;  // ready for the next call
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          const size_t seg0 = static_cast<size_t>(q + si.c0);
          const int nsg = si.nseg;
          // pass 1: per head, online max/sum over the pair's segments; lane
          // handles head lane % G of segments lane / G, lane / G + 32 / G, ...
          float rm = -INFINITY, rl = 0.f;
          for (int i = lane; i < nsg * G; i += 32) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + seg0 * G + i);
            if (ml.x != -INFINITY) {
              const float mn = fmaxf(rm, ml.x);
              rl = rl * exp2f(rm - mn) + ml.y * exp2f(ml.x - mn);
              rm = mn;
            }
          }
          for (int off = G; off < 32; off <<= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, rm, off);
            const float ol = __shfl_xor_sync(0xffffffffu, rl, off);
            const float mn = fmaxf(rm, om);
            if (mn != -INFINITY) {
              rl = (rm == -INFINITY ? 0.f : rl * exp2f(rm - mn)) + (om == -INFINITY ? 0.f : ol * exp2f(om - mn));
              rm = mn;
            }
          }
          __syncwarp();
          if (lane < G) {
            eml[lane] = rm;
            eml[kMaxGroup + lane] = rl;
          }
          __syncwarp();
          // pass 2: weighted sum of the partial outputs (independent loads)
          for (int it = lane; it < G * D4; it += 32) {
            const int g = it / D4, d = (it % D4) * 4;
            const float M = eml[g], Ls = eml[kMaxGroup + g];
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M != -INFINITY) {
              for (int sg = 0; sg < nsg; ++sg) {
                const size_t row = (seg0 + sg) * G + g;
                const float mseg = __ldcg(p.ws_ml + row * 2);
                const float4 v = __ldcg(reinterpret_cast<const float4*>(p.ws_o + row * D + d));
                const float f = mseg == -INFINITY ? 0.f : exp2f(mseg - M);
                acc.x += v.x * f;
                acc.y += v.y * f;
                acc.z += v.z * f;
                acc.w += v.w * f;
              }
            }
            const float inv = Ls > 0.f ? p.out_scale / Ls : 0.f;
            uint2 pk;
            pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(out_pair + g * D + d) = pk;
          }
        }
      }
    }
    if (*abort_flag && lane == 0 && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
    return;
  }

  // ============================== consumers ==============================
  const int c = lane & 3;    // column pair: heads 2c, 2c + 1
  const int r = lane >> 2;   // row within an 8-row group
  const int key0 = warp * 16;
  const uint8_t* stage_base = smem + L::stages;
  // 8-bit pools: the 16 keys of a step in the order m -> perm(m) (see the top)
  auto perm = [](int m) { return (m & 8) | ((m >> 1) & 3) | ((m & 1) << 2); };
  // 8-bit pools: a lane's V words cover 16-dimension chunk x (r < 4) or x + NX
  // (r >= 4) for x < NX = D / 32, i.e. exactly the D dimensions; d-tiles of P.V
  constexpr int NX = F8 ? D / 32 : 1;
  constexpr int NT = F8 ? 2 * NX : DK;

  // 8-bit pools: this lane's shared-memory offsets inside a stage's K and V
  // boxes (see the loads below), fixed for the whole kernel.  Key rows c + 4i
  // repeat their swizzle every two steps of i, 1024 bytes apart.
  uint32_t koff[F8 ? (DK + 1) / 2 : 1], voff[F8 ? 2 : 1][NX];
  if constexpr (F8) {
    const int kkey = key0 + perm(((lane >> 3) & 1) * 8 + (lane & 7));
#pragma unroll
    for (int jp = 0; jp < (DK + 1) / 2; ++jp) koff[jp] = swz128(kkey, 2 * jp + (lane >> 4));
#pragma unroll
    for (int par = 0; par < 2; ++par)
#pragma unroll
      for (int x = 0; x < NX; ++x) voff[par][x] = swz128(key0 + c + 4 * par, x + NX * (r >> 2)) + 4 * (r & 3);
  }

  uint32_t qf[DK][2];
  float o[NT][4];
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  int nseg_done = 0;

  for (int k = 0;; ++k) {
    const int s = k % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(full_bar + s), (k / kStages) & 1, abort_flag))) break;
    const StageInfo si = info[s];
    if (si.flags & kEnd) {  // pass the end on to the epilogue
      const int slot = nseg_done & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(slot_empty + slot), ((nseg_done >> 1) & 1) ^ 1, abort_flag))) break;
      if (warp == 0 && lane == 0) slot_info[slot] = si;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(slot_full + slot));
      break;
    }
    if (si.flags & kSegFirst) {
      const uint16_t* qs = reinterpret_cast<const uint16_t*>(smem + L::qbuf + size_t(s) * L::kQBytes);
      const bool gv = r < G;
#pragma unroll
      for (int kk = 0; kk < DK; ++kk) {
        if constexpr (F8) {  // dimensions 16kk + 4c .. 4c + 3 as f16 pairs
          const uint2 w = gv ? *reinterpret_cast<const uint2*>(qs + r * D + kk * 16 + 4 * c) : make_uint2(0u, 0u);
          qf[kk][0] = bf16x2_to_f16x2(w.x);
          qf[kk][1] = bf16x2_to_f16x2(w.y);
        } else {
          qf[kk][0] = gv ? *reinterpret_cast<const uint32_t*>(qs + r * D + kk * 16 + 2 * c) : 0u;
          qf[kk][1] = gv ? *reinterpret_cast<const uint32_t*>(qs + r * D + kk * 16 + 8 + 2 * c) : 0u;
        }
      }
#pragma unroll
      for (int dt = 0; dt < NT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
      m_a = m_b = -INFINITY;
      l_a = l_b = 0.f;
    }
    const bool work = si.khi > si.klo && si.klo < key0 + 16 && si.khi > key0;
    constexpr int KR = F8 ? (DK + 1) / 2 : DK;  // ldmatrix.x4 of K per step
    constexpr int VR = F8 ? NX : DK;            // V fragments per step
    uint32_t ka[KR][4], va[VR][4];
    if (work) {
      const uint8_t* kbuf = stage_base + size_t(s) * L::kStageBytes;
      const uint8_t* vbuf = kbuf + NB * kBoxBytes;
      if (si.klo > key0 || si.khi < key0 + 16) {
        // Partial slice: zero the value rows of masked keys so that stale or
        // uninitialised pool contents (possibly NaN) cannot reach P.V.
        uint8_t* vw = const_cast<uint8_t*>(vbuf);
        for (int i = lane; i < 16 * NB * 8; i += 32) {
          const int row = i / (NB * 8);
          const int rest = i % (NB * 8);
          const int key = key0 + row;
          if (key < si.klo || key >= si.khi)
            *reinterpret_cast<uint4*>(vw + (rest >> 3) * kBoxBytes + key * 128 + (rest & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const uint32_t kaddr = smem_addr(kbuf);
      const uint32_t vaddr = smem_addr(vbuf);
      if constexpr (F8) {
        // K: lane L addresses key perm(m) of matrix row m = ((L >> 3) & 1) * 8 + (L & 7),
        // 16-byte chunk 2 * jp + (L >> 4)
#pragma unroll
        for (int jp = 0; jp < KR; ++jp) ldsm_x4(kaddr + koff[jp], ka[jp][0], ka[jp][1], ka[jp][2], ka[jp][3]);
        // V: words of keys c + 4i, dimensions 16 * chunk + 4 * (r & 3) .. + 3,
        // chunk x for r < 4 and x + NX for r >= 4 (no bank conflicts when the two
        // chunks lie in different halves of the 128-byte swizzle, as for D = 128)
#pragma unroll
        for (int x = 0; x < NX; ++x)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            va[x][i] = *reinterpret_cast<const uint32_t*>(vbuf + voff[i & 1][x] + 1024 * (i >> 1));
      } else {
        const int kkey = key0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int vkey = key0 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int kk = 0; kk < DK; ++kk) {
          const int chunk = kk * 2 + (lane >> 4);
          ldsm_x4(kaddr + (chunk >> 3) * kBoxBytes + swz128(kkey, chunk & 7), ka[kk][0], ka[kk][1], ka[kk][2],
                  ka[kk][3]);
        }
#pragma unroll
        for (int dt = 0; dt < DK; ++dt) {
          const int chunk = dt * 2 + ((lane >> 3) & 1);
          ldsm_x4_trans(vaddr + (chunk >> 3) * kBoxBytes + swz128(vkey, chunk & 7), va[dt][0], va[dt][1],
                        va[dt][2], va[dt][3]);
        }
      }
    }
    // the fragments are in registers: release the stage before the math
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(empty_bar + s));

    if (work) {
      // ---- S^T = K Q^T (two independent accumulation chains) ----
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (F8) {
#pragma unroll
        for (int kk = 0; kk < DK; ++kk) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(ka[kk >> 1][(kk & 1) * 2], a0, a2);
          e4m3x4_to_f16x2x2(ka[kk >> 1][(kk & 1) * 2 + 1], a1, a3);
          mma_f16_16816((kk & 1) ? sd : sc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < DK; kk += 2) {
          mma_bf16_16816(sc, ka[kk][0], ka[kk][1], ka[kk][2], ka[kk][3], qf[kk][0], qf[kk][1]);
          if (kk + 1 < DK)
            mma_bf16_16816(sd, ka[kk + 1][0], ka[kk + 1][1], ka[kk + 1][2], ka[kk + 1][3], qf[kk + 1][0],
                           qf[kk + 1][1]);
        }
      }
      // ---- mask, online softmax (log2 domain) ----
      const int kr0 = key0 + (F8 ? perm(r) : r), kr1 = kr0 + 8;
      const bool v0 = kr0 >= si.klo && kr0 < si.khi;
      const bool v1 = kr1 >= si.klo && kr1 < si.khi;
      const float s0 = v0 ? (sc[0] + sd[0]) * p.scale_log2 : -INFINITY;
      const float s1 = v0 ? (sc[1] + sd[1]) * p.scale_log2 : -INFINITY;
      const float s2 = v1 ? (sc[2] + sd[2]) * p.scale_log2 : -INFINITY;
      const float s3 = v1 ? (sc[3] + sd[3]) * p.scale_log2 : -INFINITY;
      float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
      }
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      // no running max of the warp moved: O needs no rescaling (alpha = 1)
      const bool same_max = __all_sync(0xffffffffu, mn_a == m_a && mn_b == m_b);
      const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
      const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
      const float al_a = ex2_approx(m_a - base_a), al_b = ex2_approx(m_b - base_b);
      const float p0 = ex2_approx(s0 - base_a), p1 = ex2_approx(s1 - base_b);
      const float p2 = ex2_approx(s2 - base_a), p3 = ex2_approx(s3 - base_b);
      l_a = l_a * al_a + (p0 + p2);
      l_b = l_b * al_b + (p1 + p3);
      m_a = mn_a;
      m_b = mn_b;
      // ---- O^T = O^T * alpha + V^T P^T ----
      if constexpr (F8) {
        const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2, p3));
        if (!same_max) {
#pragma unroll
          for (int dt = 0; dt < NT; ++dt) {
            o[dt][0] *= al_a;
            o[dt][1] *= al_b;
            o[dt][2] *= al_a;
            o[dt][3] *= al_b;
          }
        }
#pragma unroll
        for (int x = 0; x < NX; ++x) {
          // bytes (key c, key c+4) and (key c+8, key c+12) of dimensions 0,1 then 2,3
          const uint32_t e01 = __byte_perm(va[x][0], va[x][1], 0x5140);
          const uint32_t f01 = __byte_perm(va[x][2], va[x][3], 0x5140);
          const uint32_t e23 = __byte_perm(va[x][0], va[x][1], 0x7362);
          const uint32_t f23 = __byte_perm(va[x][2], va[x][3], 0x7362);
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(e01, a0, a1);
          e4m3x4_to_f16x2x2(f01, a2, a3);
          mma_f16_16816(o[2 * x], a0, a1, a2, a3, pb0, pb1);
          e4m3x4_to_f16x2x2(e23, a0, a1);
          e4m3x4_to_f16x2x2(f23, a2, a3);
          mma_f16_16816(o[2 * x + 1], a0, a1, a2, a3, pb0, pb1);
        }
      } else {
        const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
        if (!same_max) {
#pragma unroll
          for (int dt = 0; dt < DK; ++dt) {
            o[dt][0] *= al_a;
            o[dt][1] *= al_b;
            o[dt][2] *= al_a;
            o[dt][3] *= al_b;
          }
        }
#pragma unroll
        for (int dt = 0; dt < DK; ++dt)
          mma_bf16_16816(o[dt], va[dt][0], va[dt][1], va[dt][2], va[dt][3], pb0, pb1);
      }
    }

    if (si.flags & kSegLast) {
      // ---- hand this warp's state for the segment to the epilogue ----
      float la = l_a, lb = l_b;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, off);
        lb += __shfl_xor_sync(0xffffffffu, lb, off);
      }
      const int slot = nseg_done & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(slot_empty + slot), ((nseg_done >> 1) & 1) ^ 1, abort_flag))) break;
      if (lane < 4) {
        mst[(slot * kConsumerWarps + warp) * kMaxGroup + 2 * c] = m_a;
        mst[(slot * kConsumerWarps + warp) * kMaxGroup + 2 * c + 1] = m_b;
        lst[(slot * kConsumerWarps + warp) * kMaxGroup + 2 * c] = la;
        lst[(slot * kConsumerWarps + warp) * kMaxGroup + 2 * c + 1] = lb;
      }
      if (warp == 0 && lane == 0) slot_info[slot] = si;
      float* ow = ost + size_t(slot) * L::kSlotFloats + size_t(warp) * kMaxGroup * L::kOStride;
      if constexpr (F8) {
#pragma unroll
        for (int dt = 0; dt < NT; ++dt) {
          // d-tile dt: pair x = dt / 2, dimensions 0,1 (even dt) or 2,3 (odd dt) of the lane's word
          const int d = 16 * (dt / 2 + NX * (r >> 2)) + 4 * (r & 3) + 2 * (dt & 1);
          if (d < D) {
            ow[(2 * c) * L::kOStride + d] = o[dt][0];
            ow[(2 * c + 1) * L::kOStride + d] = o[dt][1];
            ow[(2 * c) * L::kOStride + d + 1] = o[dt][2];
            ow[(2 * c + 1) * L::kOStride + d + 1] = o[dt][3];
          }
        }
      } else {
#pragma unroll
        for (int dt = 0; dt < DK; ++dt) {
          ow[(2 * c) * L::kOStride + dt * 16 + r] = o[dt][0];
          ow[(2 * c + 1) * L::kOStride + dt * 16 + r] = o[dt][1];
          ow[(2 * c) * L::kOStride + dt * 16 + r + 8] = o[dt][2];
          ow[(2 * c + 1) * L::kOStride + dt * 16 + r + 8] = o[dt][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(slot_full + slot));
      ++nseg_done;
    }
  }
  if (*abort_flag && lane == 0 && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
}

template <int D, int MODE>
cudaError_t launch_decode_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                            const DecodeLaunch& launch, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(launch.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = launch.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, MODE>, kmap, vmap, p);
}

template <int D, int MODE>
cudaError_t prepare_t(int B, DecodeLaunch* launch) {
  const size_t bytes = DecodeSmem<D, MODE>::bytes(B);
  const void* fn = reinterpret_cast<const void*>(decode_kernel<D, MODE>);
  cudaError_t err = set_max_dynamic_smem(fn, static_cast<int>(bytes));
  if (err != cudaSuccess) return err;
  launch->smem_bytes = static_cast<int>(bytes);
  int per_sm = 1;
  if (MODE != kModeBf16) {  // two CTAs per SM when they fit (shared memory grows with B)
    err = occupancy_blocks(&per_sm, fn, kThreads, bytes);
    if (err != cudaSuccess) return err;
    per_sm = per_sm >= 2 ? 2 : 1;
  }
  launch->grid = device_sm_count() * per_sm;
  launch->mode = MODE;
  return cudaSuccess;
}

}  // namespace

DecodeWorkspace decode_workspace_layout(int rows, int hkv, int group, int head_dim, int grid) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  DecodeWorkspace w;
  const size_t segs = static_cast<size_t>(rows) * hkv + static_cast<size_t>(kChunksPerCta) * grid;
  w.next = 0;
  w.count = 256;
  w.ml = up(w.count + static_cast<size_t>(rows) * hkv * 4);
  w.o = up(w.ml + segs * group * 2 * 4);
  w.total = up(w.o + segs * group * static_cast<size_t>(head_dim) * 4);
  return w;
}

cudaError_t decode_prepare(int head_dim, bool kv8, int B, int hkv, DecodeLaunch* launch, bool fused) {
  // bf16 pools: two CTAs per SM (twice the warps, finer pieces) when there are
  // at least two (row, kv head) pairs per CTA of that grid, so that few pairs
  // are cut between CTAs; fewer pairs keep one CTA per SM and deeper rings.
  // The one-kernel decode step takes two CTAs per SM as well: the next step's
  // CTAs then fit beside this step's and run their prologue early.
  const int mode = kv8 ? kModeE4m3
                       : (fused || static_cast<long long>(B) * hkv >= 4ll * device_sm_count() ? kModeBf16Two
                                                                                               : kModeBf16);
  switch (head_dim * 4 + mode) {
    case 256: return prepare_t<64, kModeBf16>(B, launch);
    case 257: return prepare_t<64, kModeBf16Two>(B, launch);
    case 258: return prepare_t<64, kModeE4m3>(B, launch);
    case 384: return prepare_t<96, kModeBf16>(B, launch);
    case 385: return prepare_t<96, kModeBf16Two>(B, launch);
    case 386: return prepare_t<96, kModeE4m3>(B, launch);
    case 512: return prepare_t<128, kModeBf16>(B, launch);
    case 513: return prepare_t<128, kModeBf16Two>(B, launch);
    case 514: return prepare_t<128, kModeE4m3>(B, launch);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                          int head_dim, const DecodeLaunch& launch, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  switch (head_dim * 4 + launch.mode) {
    case 256: return launch_decode_t<64, kModeBf16>(kmap, vmap, p, launch, stream);
    case 257: return launch_decode_t<64, kModeBf16Two>(kmap, vmap, p, launch, stream);
    case 258: return launch_decode_t<64, kModeE4m3>(kmap, vmap, p, launch, stream);
    case 384: return launch_decode_t<96, kModeBf16>(kmap, vmap, p, launch, stream);
    case 385: return launch_decode_t<96, kModeBf16Two>(kmap, vmap, p, launch, stream);
    case 386: return launch_decode_t<96, kModeE4m3>(kmap, vmap, p, launch, stream);
    case 512: return launch_decode_t<128, kModeBf16>(kmap, vmap, p, launch, stream);
    case 513: return launch_decode_t<128, kModeBf16Two>(kmap, vmap, p, launch, stream);
    case 514: return launch_decode_t<128, kModeE4m3>(kmap, vmap, p, launch, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lnk
