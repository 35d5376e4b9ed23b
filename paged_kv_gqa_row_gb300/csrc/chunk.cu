// K4: packed prompt chunks (prefill_paged / the prompt part of step_paged) on
// the fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Every chunk token attends over its own row's pages up to its position (and
// the window).  A CTA takes one tile of consecutive pack tokens and one kv
// head: 256 / G tokens times the G query heads of that kv head, i.e. 256
// query rows (row m = token * G + head) in two halves of 128 rows; each half
// owns the 128 tensor-memory lanes in its own 256 columns.  Tokens of a tile
// are grouped into runs of equal table rows; for each run the pages covering
// the run's key range are streamed through the kernel once, for both halves.
//
// CTA structure (320 threads, warp-specialised):
//  * warp 0, producer: loads each page's K and V (2-D TMA boxes, 128-byte
//    swizzle) into a ring of stages;
//  * warp 1, MMA: one thread issues, per page j and half h,
//      S_h[128 x 64]  = Q_h K_j^T        (tcgen05.mma; Q_h from tensor memory,
//                                         K_j K-major in shared memory)
//      O_h[128 x D]  += P_h V_j          (P from tensor memory as bf16, written
//                                         over the first 32 columns of S_h;
//                                         V_j MN-major in shared memory)
//    in the order P.V of half 0, Q.K of half 0 for the next page, then the
//    same for half 1: while the softmax of one half works on a page the
//    tensor core serves the other half (ping-pong).  The products issued by
//    one thread run in order, so Q.K of the next page overwrites S_h only
//    after P.V has read P from it.  With Q in tensor memory a Q.K product
//    reads only K from shared memory;
//  * warps 2-9, softmax, four per half: thread r of a half owns query row r
//    (tensor-memory lane r).  It first writes its query row into tensor
//    memory; then, per page, it reads its 64 scores, masks them (same run,
//    lo <= key <= position), updates the running max and sum in registers,
//    writes P back to tensor memory, and rescales its row of O only when the
//    running max grows by more than 2^8 (until then P stays below 256, exact
//    enough in bf16); at the end it normalises its row of O and stores it.
//
// Sources: "Mistral 7B Instruct v0.3", Entries table (prefill_paged: prompts
// packed end to end, each token written at its place in the pool and attending
// over its row's pages up to its position; step_paged); "Phi-3 Mini 4K
// Instruct -- files", src/attention.linnet (prefill_packed / step_packed:
// rows, positions, segments; window_mask; scale rsqrt(head_dim)).
#include "common.cuh"
#include "ptx.cuh"

namespace lnk {
namespace {

constexpr int kHalves = kChunkHalves;
constexpr int kSoftmaxWarps = 4 * kHalves;
constexpr int kThreads = (2 + kSoftmaxWarps) * 32;
constexpr int kStages = 4;
constexpr int kRows = 128;                // query rows per half = tensor-memory lanes
constexpr int kTileRows = kRows * kHalves;
constexpr float kRescaleLog2 = 8.f;       // rescale O when the max grows by more than 2^8
constexpr int kMaxOrderedTiles = 512;     // tiles ordered by cost (larger launches keep token order)

struct PageInfo {
  int run, key_base, valid, pad;
};

template <int D>
struct TcSmem {
  static constexpr int NB = boxes_for(D);
  static constexpr int kStageBytes = 2 * NB * kBoxBytes;    // K boxes, then V boxes
  static constexpr int kPvN = D <= 64 ? 64 : 128;           // N of the P.V product (D = 96 padded)
  static constexpr uint32_t kTmemCols = 512;
  // tensor-memory columns of a half (half h adds h * kHalfCols): Q (bf16
  // pairs), S (P of the page over its first 32 columns), O
  static constexpr uint32_t kHalfCols = 256;
  static constexpr uint32_t kColQ = 0, kColS = 64, kColO = 128;
  static constexpr size_t stages = 0;
  static constexpr size_t bars = stages + size_t(kStages) * kStageBytes;
  // full[S], empty[S], q_full, s_full[H], p_full[H], pv_done[H], zero
  static constexpr int kNumBars = 2 * kStages + 2 + 3 * kHalves;
  static constexpr size_t info = bars + kNumBars * sizeof(uint64_t);
  static constexpr size_t tok = info + kStages * sizeof(PageInfo);
  static constexpr size_t runs = tok + 4 * kTileRows * 4;
  static constexpr size_t misc = runs + 4 * kTileRows * 4;  // [0] runs, [1] pages, [2] abort, [3] tmem base, [4] tile
  static constexpr size_t cost = misc + 64;                   // [kMaxOrderedTiles] estimated pages per tile
  static constexpr size_t end = cost + kMaxOrderedTiles * 4;
  // more than half of the shared memory, so that one CTA holds the tensor memory of an SM
  static constexpr size_t bytes = (end + 1024) > 120 * 1024 ? (end + 1024) : 120 * 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const ChunkParams p) {
  using L = TcSmem<D>;
  constexpr int NB = L::NB;
  constexpr int DK = D / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* q_full = empty_bar + kStages;
  uint64_t* s_full = q_full + 1;          // [H]
  uint64_t* p_full = s_full + kHalves;    // [H]
  uint64_t* pv_done = p_full + kHalves;   // [H]
  uint64_t* zero_bar = pv_done + kHalves;
  PageInfo* info = reinterpret_cast<PageInfo*>(smem + L::info);
  int* tok_lo = reinterpret_cast<int*>(smem + L::tok);
  int* tok_hi = tok_lo + kTileRows;
  int* tok_run = tok_hi + kTileRows;
  int* tok_row = tok_run + kTileRows;
  int* run_row = reinterpret_cast<int*>(smem + L::runs);
  int* run_kmin = run_row + kTileRows;
  int* run_kmax = run_kmin + kTileRows;
  int* run_pages = run_kmax + kTileRows;
  int* misc = reinterpret_cast<int*>(smem + L::misc);
  volatile int* abort_flag = misc + 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.group;
  const int TQ = kHalves * p.tile_tokens;  // tokens of the tile
  // Longest tiles first: CTAs are dispatched in launch order, so the CTA of
  // launch rank L takes the (L / Hkv)-th tile by estimated cost (pages up to
  // its last position) and kv head L % Hkv.  Every CTA computes the same order.
  int tile, h;
  if (p.num_tiles <= kMaxOrderedTiles) {
    int* cost = reinterpret_cast<int*>(smem + L::cost);
    for (int i = tid; i < p.num_tiles; i += kThreads) {
      const int a = p.positions[i * TQ], b = p.positions[min(p.P, (i + 1) * TQ) - 1];
      const int pm = max(a, b);
      cost[i] = pm >= 0 ? pm / kPage + 1 : 0;
    }
    __syncthreads();
    const int rank_wanted = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x) / p.hkv;
    for (int i = tid; i < p.num_tiles; i += kThreads) {
      const int ci = cost[i];
      int rank = 0;
      for (int k = 0; k < p.num_tiles; ++k) {
        const int ck = cost[k];
        rank += (ck > ci) || (ck == ci && k > i);  // ties: later tokens first
      }
      if (rank == rank_wanted) misc[4] = i;
    }
    __syncthreads();
    tile = misc[4];
    h = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x) % p.hkv;
  } else {
    tile = p.num_tiles - 1 - static_cast<int>(blockIdx.x);  // later tokens first
    h = blockIdx.y;
  }
  const int t0 = tile * TQ;
  const int nt = min(TQ, p.P - t0);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(full_bar + s), 1);
      mbar_init(smem_addr(empty_bar + s), 1);
    }
    mbar_init(smem_addr(q_full), kSoftmaxWarps);
    for (int i = 0; i < kHalves; ++i) {
      mbar_init(smem_addr(s_full + i), 1);
      mbar_init(smem_addr(p_full + i), 4);
      mbar_init(smem_addr(pv_done + i), 1);
    }
    mbar_init(smem_addr(zero_bar), kTileRows);
    misc[2] = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(misc + 3), L::kTmemCols);
  // ---- tokens of the tile ----
  if (tid < TQ) {
    int lo = 0, hi = 0, bad = 0, row = -1;
    if (tid < nt) {
      const int t = t0 + tid;
      const int pos = p.positions[t];
      row = p.rows[t];
      if (pos >= 0) {
        if (row < 0 || row >= p.num_rows) bad = LNK_DEV_BAD_ROW;
        else if (pos >= p.pages_per_row * kPage) bad = LNK_DEV_BAD_POSITION;
        else {
          lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
          hi = pos + 1;
        }
      }
      if (h == 0 && p.segments != nullptr && t > 0 && p.segments[t] == p.segments[t - 1] &&
          p.rows[t] != p.rows[t - 1])
        bad |= LNK_DEV_SEGMENT;
    }
    tok_lo[tid] = lo;
    tok_hi[tid] = hi;
    tok_row[tid] = row;
    if (bad && h == 0 && p.status != nullptr) atomicOr(p.status, bad);
  }
  __syncthreads();
  if (tid == 0) {
    int nr = 0, cur = -1, pages = 0;
    for (int i = 0; i < nt; ++i) {
      if (tok_hi[i] <= tok_lo[i]) {
        tok_run[i] = -1;
        continue;
      }
      const int row = tok_row[i];
      if (cur < 0 || run_row[cur] != row) {
        cur = nr++;
        run_row[cur] = row;
        run_kmin[cur] = tok_lo[i];
        run_kmax[cur] = tok_hi[i];
      } else {
        run_kmin[cur] = min(run_kmin[cur], tok_lo[i]);
        run_kmax[cur] = max(run_kmax[cur], tok_hi[i]);
      }
      tok_run[i] = cur;
    }
    for (int i = nt; i < TQ; ++i) tok_run[i] = -1;
    for (int r = 0; r < nr; ++r) {
      run_pages[r] = (run_kmax[r] - 1) / kPage - run_kmin[r] / kPage + 1;
      pages += run_pages[r];
    }
    misc[0] = nr;
    misc[1] = pages;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nruns = misc[0];
  const int npages = misc[1];
  const uint32_t tmem = static_cast<uint32_t>(misc[3]);

  if (warp == 0) {
    // ============================== producer ==============================
    if (lane == 0 && npages > 0) {
      int k = 0;
      bool stop = false;
      for (int run = 0; run < nruns && !stop; ++run) {
        const int* trow = p.table + static_cast<long long>(run_row[run]) * p.pages_per_row;
        const int first = run_kmin[run] / kPage;
        for (int j = 0; j < run_pages[run]; ++j, ++k) {
          const int s = k % kStages;
          if (k >= kStages && !mbar_wait(smem_addr(empty_bar + s), ((k / kStages) - 1) & 1, abort_flag)) {
            stop = true;
            break;
          }
          const int lp = first + j;
          const int page = trow[lp];
          const uint32_t fb = smem_addr(full_bar + s);
          PageInfo si{run, lp * kPage, 1, 0};
          if (page < 0 || page >= p.num_pages) {
            if (p.status != nullptr) atomicOr(p.status, LNK_DEV_BAD_PAGE);
            si.valid = 0;
            info[s] = si;
            mbar_arrive(fb);
          } else {
            info[s] = si;
            mbar_arrive_expect_tx(fb, L::kStageBytes);
            const uint32_t kdst = smem_addr(smem + L::stages + size_t(s) * L::kStageBytes);
            const uint32_t vdst = kdst + NB * kBoxBytes;
            const int y = (h * p.num_pages + page) * kPage;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              tma_load_2d(kdst + nb * kBoxBytes, &kmap, nb * kBoxCols, y, fb);
              tma_load_2d(vdst + nb * kBoxBytes, &vmap, nb * kBoxCols, y, fb);
            }
          }
        }
      }
      // do not leave while a copy may still land in this CTA's memory
      const int issued = k;
      for (int kk = max(0, issued - kStages); kk < issued; ++kk) {
        const uint32_t fb = smem_addr(full_bar + kk % kStages);
        const uint64_t t_0 = global_timer_ns();
        while (!mbar_try_wait(fb, (kk / kStages) & 1) && global_timer_ns() - t_0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ================================ MMA =================================
    if (lane == 0 && npages > 0) {
      constexpr uint32_t kIdS = umma_idesc_bf16(kRows, 64, 0, 0);
      constexpr uint32_t kIdPV = umma_idesc_bf16(kRows, L::kPvN, 0, 1);
      // Descriptors of stage 0's K (K-major) and V (MN-major) boxes; another
      // stage or K step adds its byte offset / 16 to the 14-bit address field,
      // which cannot carry (shared addresses stay below 256 KiB).
      const uint32_t stage0 = smem_addr(smem + L::stages);
      const uint64_t kdesc0 = umma_desc_sw128(stage0, 0, 1024);
      const uint64_t vdesc0 = umma_desc_sw128(stage0 + NB * kBoxBytes, kBoxBytes, 1024);
      // S_hf = Q_hf K^T for the page in stage s (Q from tensor memory)
      auto issue_s = [&](int hf, int s) {
        const uint64_t kd = kdesc0 + static_cast<uint64_t>((s * L::kStageBytes) >> 4);
        const uint32_t hc = tmem + hf * L::kHalfCols;
#pragma unroll
        for (int kk = 0; kk < DK; ++kk) {
          const uint64_t bd = kd + (((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          umma_ts(hc + L::kColS, hc + L::kColQ + kk * 8, bd, kIdS, kk > 0);
        }
        umma_commit(smem_addr(s_full + hf));
      };
      bool ok = mbar_wait(smem_addr(q_full), 0, abort_flag) && mbar_wait(smem_addr(full_bar), 0, abort_flag);
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf) issue_s(hf, 0);
      }
      int last_pv = -1;
      for (int j = 0; ok && j < npages; ++j) {
        const int s = j % kStages;
        const uint64_t vd = vdesc0 + static_cast<uint64_t>((s * L::kStageBytes) >> 4);
#pragma unroll
        for (int hf = 0; hf < kHalves && ok; ++hf) {
          ok = mbar_wait(smem_addr(p_full + hf), j & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t hc = tmem + hf * L::kHalfCols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 64 keys, 16 per instruction
            const uint64_t bd = vd + ((kk * 16 * 128) >> 4);
            umma_ts(hc + L::kColO, hc + L::kColS + kk * 8, bd, kIdPV, (j > 0 || kk > 0));
          }
          umma_commit(smem_addr(pv_done + hf));
          if (hf == kHalves - 1) {
            umma_commit(smem_addr(empty_bar + s));
            last_pv = j;
          }
          if (j + 1 < npages) {
            const int s1 = (j + 1) % kStages;
            if (hf == 0) {
              ok = mbar_wait(smem_addr(full_bar + s1), ((j + 1) / kStages) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(hf, s1);
          }
        }
      }
      // the tensor memory is freed at the end: let the last products finish
      if (last_pv >= 0) {
        for (int hf = 0; hf < kHalves; ++hf) {
          const uint32_t bar = smem_addr(pv_done + hf);
          const uint64_t t_0 = global_timer_ns();
          while (!mbar_try_wait(bar, last_pv & 1) && global_timer_ns() - t_0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else {
    // ============================== softmax ===============================
    const int hf = (warp - 2) / 4;        // half of the tile
    const int qt = warp & 3;              // tensor-memory lane quarter of this warp
    const int row = hf * kRows + qt * 32 + lane;  // query row of the tile = token * G + head
    const int tl = row / G, g = row % G;
    const int lo = tok_lo[tl], hi = tok_hi[tl], run_id = tok_run[tl];
    const bool live = tl < nt && run_id >= 0;
    const uint32_t hcol = tmem + (static_cast<uint32_t>(qt * 32) << 16) + hf * L::kHalfCols;
    const int ctid = tid - 64;            // 0..255 among the softmax threads
    const size_t qrow = (static_cast<size_t>(t0 + tl) * p.hq + static_cast<size_t>(h) * G + g) * D;
    // ---- this row's query into tensor memory (bf16 pairs, the A operand of Q.K) ----
    if (npages > 0) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {  // 8 bf16 pairs = two 16-byte loads per step
        uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
        if (tl < nt) {
          a = src[2 * c];
          b = src[2 * c + 1];
        }
        const uint32_t r[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        tmem_st8(hcol + L::kColQ + c * 8, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(q_full));
    }
    // Every wait's outcome is made warp-uniform: the tensor-memory loads and
    // stores that follow are warp-collective.
    float m_ref = -INFINITY, l_sum = 0.f;
    uint32_t zero_uses = 0;
    bool ok = true;
    for (int j = 0; j < npages && ok; ++j) {
      const int s = j % kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(full_bar + s), (j / kStages) & 1, abort_flag));
      if (!ok) break;
      const PageInfo si = info[s];
      const int kmin = run_kmin[si.run], kmax = run_kmax[si.run];
      if (!si.valid || si.key_base < kmin || si.key_base + kPage > kmax) {
        // Keys of this page outside the run's range may hold stale or
        // uninitialised data: zero their value rows before P.V reads them.
        uint8_t* vb = smem + L::stages + size_t(s) * L::kStageBytes + NB * kBoxBytes;
        for (int i = ctid; i < kPage * NB * 8; i += kTileRows) {
          const int key = i / (NB * 8), rest = i % (NB * 8);
          if (!si.valid || si.key_base + key < kmin || si.key_base + key >= kmax)
            *reinterpret_cast<uint4*>(vb + (rest >> 3) * kBoxBytes + key * 128 + (rest & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_addr(zero_bar));
        ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(zero_bar), zero_uses & 1u, abort_flag));
        ++zero_uses;
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(s_full + hf), j & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float x[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(hcol + L::kColS, r0);
        tmem_ld32(hcol + L::kColS + 32, r1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(r0[i]);
          x[32 + i] = __uint_as_float(r1[i]);
        }
      }
      // visible keys of this page for this row: [ka, ke)
      const bool in_run = live && si.valid && si.run == run_id;
      const int ka = in_run ? max(lo - si.key_base, 0) : kPage;
      const int ke = in_run ? max(ka, min(hi - si.key_base, kPage)) : kPage;
      if (!__all_sync(0xffffffffu, ka == 0 && ke == kPage)) {
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = (i >= ka && i < ke) ? x[i] : -INFINITY;
      }
      // row max as a tree of independent maxima
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = fmaxf(x[i], x[i + 8]);
#pragma unroll
      for (int i = 16; i < 64; i += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], x[i + k]);
      const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mx = mraw == -INFINITY ? -INFINITY : mraw * p.scale_log2;  // log2 units
      // running max: rescale O only when it grows by more than 2^8
      float alpha = 1.f;
      if (mx != -INFINITY) {
        if (m_ref == -INFINITY) {
          m_ref = mx;
        } else if (mx > m_ref + kRescaleLog2) {
          alpha = exp2f(m_ref - mx);
          m_ref = mx;
          l_sum *= alpha;
        }
      }
      if (__any_sync(0xffffffffu, alpha != 1.f) && j >= 1) {
        // P.V of page j - 1
        ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(pv_done + hf), (j - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < L::kPvN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(hcol + L::kColO + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(hcol + L::kColO + c * 32, r);
        }
        tmem_st_wait();
      }
      // probabilities 2^(s * scale * log2(e) - m_ref), packed to bf16
      const float nbase = m_ref == -INFINITY ? 0.f : -m_ref;
      uint32_t pk[32];
      float r8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) r8[k] = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float e0 = ex2_approx(__fmaf_rn(x[2 * i], p.scale_log2, nbase));
        const float e1 = ex2_approx(__fmaf_rn(x[2 * i + 1], p.scale_log2, nbase));
        r8[i & 7] += e0 + e1;
        pk[i] = pack_bf16x2(e0, e1);
      }
      l_sum += ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
      tmem_st32(hcol + L::kColS, pk);  // P over the scores just read
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(p_full + hf));
    }
    // ---- normalise and store this row ----
    if (ok && npages > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(pv_done + hf), (npages - 1) & 1, abort_flag));
      tc_fence_after();
    }
    uint16_t* dst = p.out + qrow;
    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll 1
    for (int c = 0; c < L::kPvN / 16; ++c) {
      uint32_t r[16];
      if (ok && npages > 0) {
        tmem_ld16(hcol + L::kColO + c * 16, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = 0u;
      }
      if (tl < nt && c * 16 < D) {
        uint2* o = reinterpret_cast<uint2*>(dst + c * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a0 = live ? __uint_as_float(r[4 * i]) * inv : 0.f;
          const float a1 = live ? __uint_as_float(r[4 * i + 1]) * inv : 0.f;
          const float a2 = live ? __uint_as_float(r[4 * i + 2]) * inv : 0.f;
          const float a3 = live ? __uint_as_float(r[4 * i + 3]) * inv : 0.f;
          o[i] = make_uint2(pack_bf16x2(a0, a1), pack_bf16x2(a2, a3));
        }
      }
    }
  }
  if (*abort_flag && lane == 0 && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, L::kTmemCols);
}

template <int D>
cudaError_t launch_chunk_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const ChunkParams& p,
                           cudaStream_t stream) {
  const int bytes = static_cast<int>(TcSmem<D>::bytes);
  cudaError_t err = set_max_dynamic_smem(reinterpret_cast<const void*>(chunk_kernel<D>), bytes);
  if (err != cudaSuccess) return err;
  dim3 grid(p.num_tiles, p.hkv);
  chunk_kernel<D><<<grid, kThreads, bytes, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

__global__ void gather_last_kernel(const uint16_t* out, const int32_t* last, uint16_t* last_out, int P,
                                   int row_elems, int32_t* status) {
  const int m = blockIdx.x;
  const int t = last[m];
  const bool ok = t >= 0 && t < P;
  if (!ok && threadIdx.x == 0 && status != nullptr) atomicOr(status, LNK_DEV_BAD_LAST);
  for (int i = threadIdx.x; i < row_elems; i += blockDim.x)
    last_out[static_cast<size_t>(m) * row_elems + i] = ok ? out[static_cast<size_t>(t) * row_elems + i] : 0;
}

}  // namespace

cudaError_t launch_chunk(const CUtensorMap& kmap, const CUtensorMap& vmap, const ChunkParams& p, int head_dim,
                         cudaStream_t stream) {
  if (p.P == 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch_chunk_t<64>(kmap, vmap, p, stream);
    case 96: return launch_chunk_t<96>(kmap, vmap, p, stream);
    case 128: return launch_chunk_t<128>(kmap, vmap, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gather_last(const uint16_t* out, const int32_t* last, uint16_t* last_out, int M, int P,
                               int row_elems, int32_t* status, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  gather_last_kernel<<<M, 256, 0, stream>>>(out, last, last_out, P, row_elems, status);
  return cudaGetLastError();
}

}  // namespace lnk
