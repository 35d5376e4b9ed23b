// K4: packed prompt chunks (prefill_paged / the prompt part of step_paged) on
// the fifth-generation tensor cores, two SMs per tile (tcgen05 cta_group::2,
// accumulators in tensor memory).
//
// Every chunk token attends over its own row's pages up to its position (and
// the window).  A tile is 256 / G consecutive pack tokens times the G query
// heads of one kv head: 256 query rows (row m = token * G + head).  A cluster
// of two CTAs takes one tile: CTA rank r owns rows 128 r .. 128 r + 127 in its
// tensor-memory lanes.  Tokens of a tile are grouped into runs of equal table
// rows; the pages covering each run's key range are streamed once, two pages
// (128 keys) per step, for all 256 rows.
//
// Products are 2-SM (M = 256), issued by two threads of rank 0:
//   S_b[256 x 128] = Q K_j^T   Q K-major in each CTA's shared memory (its 128
//                              rows), K_j K-major in shared memory: rank r
//                              holds page 2j + r of the step (keys
//                              64 r .. 64 r + 63);
//   O[256 x 128]  += P_b V_j   P_b from tensor memory (bf16 pairs), V_j
//                              MN-major: rank r holds head-dim columns
//                              64 r .. 64 r + 63 of both pages.
// S and P are double-buffered (b = j mod 2), so Q K^T of step j + 1 runs on
// the tensor cores while the softmax works on step j.
//
// CTA structure (352 threads, warp-specialised, both ranks):
//  * warp 0, producer: TMA loads of this CTA's K page and V columns into
//    rings of stages (and, before that, the tile's runs of tokens);
//  * warp 1: in rank 0, the Q.K^T issuer; in rank 1, a relay that tells rank
//    0 when rank 1's stages have landed (rank 0's products read both CTAs'
//    stages);
//  * warp 10: in rank 0, the P.V issuer;
//  * warps 2-9, softmax, in two groups of four warps taking alternate steps:
//    thread r of a group owns query row r of its CTA (tensor-memory lane r).
//    The first group loads the CTA's query rows into shared memory at the
//    start.  Per step, a group reads 128 scores, masks them (same run,
//    lo <= key <= position, valid page), updates the running max (handed on
//    to the other group) and its partial sum, writes P, and rescales its row
//    of O only when the running max grows by more than 2^8 (until then P stays
//    below 256, exact enough in bf16); at the end the groups combine their
//    sums and each normalises and stores half of the row of O.
// Barriers that the other CTA arrives on live in rank 0 (the P and relay
// barriers); the 2-SM commits arrive in both CTAs at once.
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

constexpr int kThreads = 11 * 32;
constexpr int kStagesK = 4;               // K ring (this CTA's page of a step)
constexpr int kStagesV = 4;               // V ring (this CTA's columns of both pages)
constexpr int kRows = 128;                // query rows per CTA = tensor-memory lanes
constexpr int kTileRows = 2 * kRows;      // rows of a tile (both CTAs)
constexpr int kStepKeys = 2 * kPage;      // keys per step
constexpr float kRescaleLog2 = 8.f;       // rescale O when the max grows by more than 2^8
constexpr int kMaxOrderedTiles = 512;     // tiles ordered by cost (larger launches keep token order)

template <int D>
struct TcSmem {
  static constexpr int NB = boxes_for(D);
  static constexpr int kKStage = NB * kBoxBytes;            // one page of K, all head-dim columns
  static constexpr int kVStage = 2 * kBoxBytes;             // both pages of V, 64 head-dim columns
  static constexpr int kPvN = 128;                          // N of P.V (head_dim padded; 64 per CTA)
  static constexpr uint32_t kTmemCols = 512;
  // tensor-memory columns: S_0, S_1 (f32 scores), P_0, P_1 (bf16 pairs), O
  static constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;
  static constexpr int kQBox = kRows * 128;                 // 128 query rows x 64 head-dim columns
  static constexpr size_t kring = 0;
  static constexpr size_t vring = kring + size_t(kStagesK) * kKStage;
  static constexpr size_t qsm = vring + size_t(kStagesV) * kVStage;  // this CTA's query rows, K-major
  static constexpr size_t bars = qsm + size_t(NB) * kQBox;
  // kfull[K], kempty[K], vfull[V], vempty[V], sfull[2], sfree[2], pfull[2], pvdone[2], odone
  static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 9;
  static constexpr size_t tok = bars + kNumBars * sizeof(uint64_t);
  static constexpr size_t runs = tok + 4 * kTileRows * 4;
  static constexpr size_t misc = runs + 5 * kTileRows * 4;  // [0] runs, [1] steps, [2] abort, [3] tmem, [4] tile
  static constexpr size_t cost = misc + 64;                 // [kMaxOrderedTiles] estimated pages per tile
  // softmax groups' hand-off: max [2][128] and ok [2][128] per step parity;
  // at the end max, sum and ok [2][128] per group
  static constexpr size_t xchg = cost + kMaxOrderedTiles * 4;
  static constexpr size_t end = xchg + 10 * kRows * 4;
  static constexpr size_t bytes = end + 1024;
};

// Walks the steps of a tile in order: run r, step s of the run (pages
// first + 2 s and first + 2 s + 1, the second one past the run's last page
// when the run has an odd number of pages).
struct StepCursor {
  int run = 0, s = 0;
  __device__ __forceinline__ void next(const int* run_steps) {
    if (++s >= run_steps[run]) {
      ++run;
      s = 0;
    }
  }
};

constexpr int kPastRun = -2147483647 - 1;  // "entry" of a page past the end of its run

// Table entries of the two pages of the step at `c` (kPastRun for a page past
// its run, and for both past the last run).
__device__ __forceinline__ void step_entries(const ChunkParams& p, const int* run_row, const int* run_first,
                                             const int* run_kmax, int nruns, const StepCursor& c, int& ea,
                                             int& eb) {
  ea = eb = kPastRun;
  if (c.run >= nruns) return;
  const int* trow = p.table + static_cast<long long>(run_row[c.run]) * p.pages_per_row;
  const int lp = run_first[c.run] + 2 * c.s;
  ea = trow[lp];
  if (lp + 1 <= (run_kmax[c.run] - 1) / kPage) eb = trow[lp + 1];
}

template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const ChunkParams p) {
  using L = TcSmem<D>;
  constexpr int NB = L::NB;
  constexpr int DK = D / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* kempty = kfull + kStagesK;
  uint64_t* vfull = kempty + kStagesK;
  uint64_t* vempty = vfull + kStagesV;
  uint64_t* sfull = vempty + kStagesV;   // [2] Q.K^T into S_b finished
  uint64_t* sfree = sfull + 2;           // [2] the softmax has read S_b (rank 0 only)
  uint64_t* pfull = sfree + 2;           // [2] P_b written (rank 0 only)
  uint64_t* pvdone = pfull + 2;          // [2] P.V from P_b finished (all but the last)
  uint64_t* odone = pvdone + 2;          // the last P.V
  int* tok_lo = reinterpret_cast<int*>(smem + L::tok);
  int* tok_hi = tok_lo + kTileRows;
  int* tok_run = tok_hi + kTileRows;
  int* tok_row = tok_run + kTileRows;
  int* run_row = reinterpret_cast<int*>(smem + L::runs);
  int* run_kmin = run_row + kTileRows;
  int* run_kmax = run_kmin + kTileRows;
  int* run_first = run_kmax + kTileRows;  // first logical page
  int* run_steps = run_first + kTileRows;
  int* misc = reinterpret_cast<int*>(smem + L::misc);
  volatile int* abort_flag = misc + 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_cta_rank();
  const int cid = static_cast<int>(blockIdx.x >> 1);  // cluster = tile and kv head
  const int G = p.group;
  const int TQ = 2 * p.tile_tokens;       // tokens of the tile
  // Longest tiles first: clusters are dispatched in launch order, so the
  // cluster of launch rank c takes the (c / Hkv)-th tile by estimated cost
  // (pages up to its last position) and kv head c % Hkv.  Every CTA computes
  // the same order.
  int tile, h;
  if (p.num_tiles <= kMaxOrderedTiles) {
    int* cost = reinterpret_cast<int*>(smem + L::cost);
    for (int i = tid; i < p.num_tiles; i += kThreads) {
      const int a = p.positions[i * TQ], b = p.positions[min(p.P, (i + 1) * TQ) - 1];
      const int pm = max(a, b);
      cost[i] = pm >= 0 ? pm / kPage + 1 : 0;
    }
    __syncthreads();
    const int rank_wanted = cid / p.hkv;
    for (int i = tid; i < p.num_tiles; i += kThreads) {
      const int ci = cost[i];
      int rk = 0;
      for (int k = 0; k < p.num_tiles; ++k) {
        const int ck = cost[k];
        rk += (ck > ci) || (ck == ci && k > i);  // ties: later tokens first
      }
      if (rk == rank_wanted) misc[4] = i;
    }
    __syncthreads();
    tile = misc[4];
  } else {
    tile = p.num_tiles - 1 - cid / p.hkv;  // later tokens first
  }
  h = cid % p.hkv;
  const int t0 = tile * TQ;
  const int nt = min(TQ, p.P - t0);

  // ---- this CTA's query rows into shared memory (K-major, 128-byte swizzle:
  // the A operand of Q.K^T), by the first softmax group right away, so that
  // the loads overlap the tile's set-up: all of a row's 16-byte pieces are
  // loaded before any is stored.  The cluster barrier below publishes them to
  // the pair's tensor cores (each thread orders its stores before the async
  // proxy first). ----
  if (warp >= 2 && warp < 6) {
    const int rl = (warp & 3) * 32 + lane;
    const int row = static_cast<int>(rank) * kRows + rl;  // token * G + head
    const int tl = row / G, g = row % G;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + (static_cast<size_t>(t0 + tl) * p.hq + static_cast<size_t>(h) * G + g) * D);
    uint4 a[D / 8];
#pragma unroll
    for (int c = 0; c < D / 8; ++c) a[c] = tl < nt ? src[c] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
      *reinterpret_cast<uint4*>(smem + L::qsm + (c >> 3) * L::kQBox + swz128(rl, c & 7)) = a[c];
    fence_proxy_async_smem();
  }

  if (tid == 0) {
    // rank 0's full barriers also count the relay's arrival for rank 1's copy
    for (int s = 0; s < kStagesK; ++s) {
      mbar_init(smem_addr(kfull + s), rank == 0 ? 2 : 1);
      mbar_init(smem_addr(kempty + s), 1);
    }
    for (int s = 0; s < kStagesV; ++s) {
      mbar_init(smem_addr(vfull + s), rank == 0 ? 2 : 1);
      mbar_init(smem_addr(vempty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(sfull + b), 1);
      mbar_init(smem_addr(sfree + b), 8);   // one softmax group (four warps) in each CTA
      mbar_init(smem_addr(pfull + b), 8);
      mbar_init(smem_addr(pvdone + b), 1);
    }
    mbar_init(smem_addr(odone), 1);
    misc[2] = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem2_alloc(smem_addr(misc + 3), L::kTmemCols);
  // ---- tokens of the tile ----
  for (int i = tid; i < TQ; i += kThreads) {
    int lo = 0, hi = 0, bad = 0, row = -1;
    if (i < nt) {
      const int t = t0 + i;
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
    tok_lo[i] = lo;
    tok_hi[i] = hi;
    tok_row[i] = row;
    if (bad && h == 0 && rank == 0 && p.status != nullptr) atomicOr(p.status, bad);
  }
  __syncthreads();
  // ---- runs: maximal groups of the tile's valid tokens (in order, skipping
  // tokens that see no key) with one table row; one warp, 32 tokens at a time ----
  if (warp == 0) {
    int nr = 0;           // runs so far
    int last_row = 0;     // row of the last valid token so far
    bool have_last = false;
    for (int base = 0; base < TQ; base += 32) {
      const int i = base + lane;
      const bool v = i < nt && tok_hi[i] > tok_lo[i];
      const int trow = tok_row[i];
      const unsigned vm = __ballot_sync(0xffffffffu, v);
      // row of the previous valid token: in this group of 32, else carried over
      const unsigned before = vm & ((1u << lane) - 1u);
      const int prev = __shfl_sync(0xffffffffu, trow, before ? 31 - __clz(before) : lane);
      const bool has_prev = before != 0u || have_last;
      const int prev_row = before ? prev : last_row;
      const bool start = v && (!has_prev || prev_row != trow);
      const unsigned sm = __ballot_sync(0xffffffffu, start);
      const int rid = nr + __popc(sm & ((2u << lane) - 1u)) - 1;  // (lane 31: all bits)
      tok_run[i] = v ? rid : -1;
      if (start) {
        run_row[rid] = trow;
        run_kmin[rid] = tok_lo[i];
        run_kmax[rid] = tok_hi[i];
      }
      __syncwarp();
      if (v && !start) {
        atomicMin(run_kmin + rid, tok_lo[i]);
        atomicMax(run_kmax + rid, tok_hi[i]);
      }
      __syncwarp();
      nr += __popc(sm);
      if (vm) {
        last_row = __shfl_sync(0xffffffffu, trow, 31 - __clz(vm));
        have_last = true;
      }
    }
    int steps = 0;
    for (int r = lane; r < nr; r += 32) {
      run_first[r] = run_kmin[r] / kPage;
      const int pages = (run_kmax[r] - 1) / kPage - run_first[r] + 1;
      run_steps[r] = (pages + 1) / 2;
      steps += run_steps[r];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) steps += __shfl_xor_sync(0xffffffffu, steps, o);
    if (lane == 0) {
      misc[0] = nr;
      misc[1] = steps;
    }
  }
  // barriers initialised and tensor memory allocated in both CTAs before any
  // thread of either uses them
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const int nsteps = misc[1];
  const uint32_t tmem = static_cast<uint32_t>(misc[3]);

  if (warp == 0) {
    // ============================== producer ==============================
    if (lane == 0 && nsteps > 0) {
      StepCursor cur;
      int ea, eb;  // table entries of the step's two pages, read one step ahead
      step_entries(p, run_row, run_first, run_kmax, misc[0], cur, ea, eb);
      int j = 0;
      for (; j < nsteps; ++j, cur.next(run_steps)) {
        const int sk = j % kStagesK, sv = j % kStagesV;
        int na, nb;
        {
          StepCursor nc = cur;
          nc.next(run_steps);
          step_entries(p, run_row, run_first, run_kmax, misc[0], nc, na, nb);
        }
        // a page past the run or a bad table entry loads page 0 instead (its
        // keys are masked and its values zeroed)
        const bool bad_a = ea >= p.num_pages || ea < 0;
        const bool bad_b = eb != kPastRun && (eb >= p.num_pages || eb < 0);
        if (rank == 0 && (bad_a || bad_b) && p.status != nullptr) atomicOr(p.status, LNK_DEV_BAD_PAGE);
        const int pa = bad_a ? 0 : ea, pb = (bad_b || eb == kPastRun) ? 0 : eb;
        if (j >= kStagesK && !mbar_wait(smem_addr(kempty + sk), ((j / kStagesK) - 1) & 1, abort_flag)) break;
        uint32_t fb = smem_addr(kfull + sk);
        mbar_arrive_expect_tx(fb, L::kKStage);
        const uint32_t kdst = smem_addr(smem + L::kring + size_t(sk) * L::kKStage);
        const int yk = (h * p.num_pages + (rank == 0 ? pa : pb)) * kPage;  // this CTA's K page
#pragma unroll
        for (int nb2 = 0; nb2 < NB; ++nb2) tma_load_2d(kdst + nb2 * kBoxBytes, &kmap, nb2 * kBoxCols, yk, fb);
        if (j >= kStagesV && !mbar_wait(smem_addr(vempty + sv), ((j / kStagesV) - 1) & 1, abort_flag)) {
          ++j;  // this step's K load was issued
          break;
        }
        fb = smem_addr(vfull + sv);
        mbar_arrive_expect_tx(fb, L::kVStage);
        const uint32_t vdst = smem_addr(smem + L::vring + size_t(sv) * L::kVStage);
        const int xv = static_cast<int>(rank) * kBoxCols;
        tma_load_2d(vdst, &vmap, xv, (h * p.num_pages + pa) * kPage, fb);
        tma_load_2d(vdst + kBoxBytes, &vmap, xv, (h * p.num_pages + pb) * kPage, fb);
        ea = na;
        eb = nb;
      }
      // do not leave while a copy may still land in this CTA's memory
      const int issued = j;
      for (int kk = max(0, issued - kStagesK); kk < issued; ++kk) {
        const uint32_t fb = smem_addr(kfull + kk % kStagesK);
        const uint64_t t_0 = global_timer_ns();
        while (!mbar_try_wait(fb, (kk / kStagesK) & 1) && global_timer_ns() - t_0 < kWaitLimitNs) {
        }
      }
      for (int kk = max(0, issued - kStagesV); kk < issued; ++kk) {
        const uint32_t fb = smem_addr(vfull + kk % kStagesV);
        const uint64_t t_0 = global_timer_ns();
        while (!mbar_try_wait(fb, (kk / kStagesV) & 1) && global_timer_ns() - t_0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (rank != 0) {
      // ============================ relay (rank 1) ==========================
      if (lane == 0 && nsteps > 0) {
        const uint32_t kfull0 = mapa_shared(smem_addr(kfull), 0);
        const uint32_t vfull0 = mapa_shared(smem_addr(vfull), 0);
        for (int j = 0; j < nsteps; ++j) {
          const int sk = j % kStagesK, sv = j % kStagesV;
          if (!mbar_wait(smem_addr(kfull + sk), (j / kStagesK) & 1, abort_flag)) break;
          mbar_arrive_remote(kfull0 + sk * 8);
          if (!mbar_wait(smem_addr(vfull + sv), (j / kStagesV) & 1, abort_flag)) break;
          mbar_arrive_remote(vfull0 + sv * 8);
        }
      }
    } else if (lane == 0 && nsteps > 0) {
      // ======================= Q.K^T issuer (rank 0) ========================
      constexpr uint32_t kIdS = umma_idesc_bf16(kTileRows, kStepKeys, 0, 0);
      // Descriptors of stage 0's K tile and of the query rows (K-major); another
      // stage or K step adds its byte offset / 16 to the 14-bit address field,
      // which cannot carry (shared addresses stay below 256 KiB).
      const uint64_t kdesc0 = umma_desc_sw128(smem_addr(smem + L::kring), 0, 1024);
      const uint64_t qdesc0 = umma_desc_sw128(smem_addr(smem + L::qsm), 0, 1024);
      // S_b = Q K^T of step j, once the softmax has read S_b of step j - 2
      // (sfree is at most one phase past that: the softmax reads S_b of step
      // j only after this product) and both CTAs' K pages have landed.  (Both
      // CTAs' query rows were stored before the cluster barrier.)
      bool ok = true;
      for (int j = 0; ok && j < nsteps; ++j) {
        const int b = j & 1, sk = j % kStagesK;
        ok = (j < 2 || mbar_wait(smem_addr(sfree + b), ((j - 2) >> 1) & 1, abort_flag)) &&
             mbar_wait(smem_addr(kfull + sk), (j / kStagesK) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sc = tmem + L::kColS + static_cast<uint32_t>(b) * kStepKeys;
        const uint64_t kd = kdesc0 + static_cast<uint64_t>((sk * L::kKStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < DK; ++kk) {
          const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          const uint32_t qoff = ((kk >> 2) * L::kQBox + (kk & 3) * 32) >> 4;
          umma2_ss(sc, qdesc0 + qoff, kd + koff, kIdS, kk > 0);
        }
        umma2_commit_both(smem_addr(sfull + b));
        umma2_commit_both(smem_addr(kempty + sk));
      }
    }
  } else if (warp == 10) {
    if (rank == 0 && lane == 0 && nsteps > 0) {
      // ========================= P.V issuer (rank 0) ========================
      // One thread issues every P.V, in step order: O accumulates in order,
      // and a finished P.V implies that every earlier one has finished.
      constexpr uint32_t kIdPV = umma_idesc_bf16(kTileRows, L::kPvN, 0, 1);
      const uint64_t vdesc0 = umma_desc_sw128(smem_addr(smem + L::vring), 0, 1024);
      bool ok = true;
      for (int j = 0; ok && j < nsteps; ++j) {
        const int b = j & 1, sv = j % kStagesV;
        ok = mbar_wait(smem_addr(pfull + b), (j >> 1) & 1, abort_flag) &&
             mbar_wait(smem_addr(vfull + sv), (j / kStagesV) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t pc = tmem + L::kColP + static_cast<uint32_t>(b) * (kStepKeys / 2);
        const uint64_t vd = vdesc0 + static_cast<uint64_t>((sv * L::kVStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kStepKeys / 16; ++kk) {  // 16 keys per product
          const uint64_t bd = vd + ((kk * 16 * 128) >> 4);
          umma2_ts(tmem + L::kColO, pc + kk * 8, bd, kIdPV, (j > 0 || kk > 0));
        }
        umma2_commit_both(smem_addr(vempty + sv));
        umma2_commit_both(smem_addr(j + 1 < nsteps ? pvdone + b : odone));
      }
    }
  } else {
    // ============================== softmax ===============================
    // Two groups of four warps take the steps in turn: group 0 (warps 2-5)
    // the even steps, group 1 (warps 6-9) the odd ones, so that one group's
    // loads and maxima overlap the other's exponentials.  Step j uses S_(j mod
    // 2), so group g always reads and writes S_g.  Warps w and w + 4 share the
    // tensor-memory lanes of quarter w % 4: thread r of each group owns query
    // row r of this CTA.  The row's running max passes from the group of step
    // j to the group of step j + 1 through shared memory (a named barrier that
    // the publisher arrives on and the receiver waits on), together with the
    // decision to go on, so a stop reaches both groups and neither waits for
    // the other in vain.
    const int grp = (warp - 2) >> 2;
    const int qt = warp & 3;              // tensor-memory lane quarter of this warp
    const int rl = qt * 32 + lane;        // row of this CTA = tensor-memory lane
    const int row = static_cast<int>(rank) * kRows + rl;  // row of the tile = token * G + head
    const int tl = row / G, g = row % G;
    const int lo = tok_lo[tl], hi = tok_hi[tl], run_id = tok_run[tl];
    const bool live = tl < nt && run_id >= 0;
    const uint32_t lanes = static_cast<uint32_t>(qt * 32) << 16;
    const int bar_pub = 1 + qt + 4 * grp;        // this group's hand-off to the other group
    const int bar_sub = 1 + qt + 4 * (grp ^ 1);  // the other group's hand-off to this one
    const int bar_fin = 9 + qt;                  // both groups, once at the end
    float* hand_m = reinterpret_cast<float*>(smem + L::xchg);         // [2 step parities][128 rows]
    int* hand_ok = reinterpret_cast<int*>(smem + L::xchg) + 2 * kRows;  // [2][128]
    float* fin_m = reinterpret_cast<float*>(smem + L::xchg) + 4 * kRows;  // [2 groups][128]
    float* fin_l = fin_m + 2 * kRows;
    int* fin_ok = reinterpret_cast<int*>(fin_l + 2 * kRows);
    const size_t qrow = (static_cast<size_t>(t0 + tl) * p.hq + static_cast<size_t>(h) * G + g) * D;
    const uint32_t pfull0 = mapa_shared(smem_addr(pfull), 0);
    // Every wait's outcome is made warp-uniform: the tensor-memory loads and
    // stores that follow are warp-collective.
    float m_ref = -INFINITY;   // the row's running max (log2 units) after this group's last step
    float m_part = -INFINITY;  // reference of this group's partial sum
    float l_part = 0.f;        // sum of this group's probabilities, relative to m_part
    bool ok = true, stuck = false;
    StepCursor cur;
    int ea = kPastRun, eb = kPastRun;  // table entries of the step's two pages, read one step ahead
    if (nsteps > 0) step_entries(p, run_row, run_first, run_kmax, misc[0], cur, ea, eb);
    const uint32_t sc = tmem + lanes + L::kColS + static_cast<uint32_t>(grp) * kStepKeys;  // S_grp
    const uint32_t pcol = tmem + lanes + L::kColP + static_cast<uint32_t>(grp) * (kStepKeys / 2);  // P_grp
    const uint32_t sfree0 = mapa_shared(smem_addr(sfree), 0);
    for (int j = 0; j < nsteps; ++j, cur.next(run_steps)) {
      const int kmin = run_kmin[cur.run], kmax = run_kmax[cur.run];
      const int lpa = run_first[cur.run] + 2 * cur.s;
      const int kb = lpa * kPage;         // logical key of the step's first slot
      // pages of the step that hold data: in the run and with a valid table entry
      const bool va = ea >= 0 && ea < p.num_pages;
      const bool vb = eb >= 0 && eb < p.num_pages;
      {
        StepCursor nc = cur;
        nc.next(run_steps);
        step_entries(p, run_row, run_first, run_kmax, misc[0], nc, ea, eb);
      }
      if ((j & 1) != grp) continue;
      const int sv = j % kStagesV;
      bool okw = !stuck && __all_sync(0xffffffffu, mbar_wait(smem_addr(sfull + grp), (j >> 1) & 1, abort_flag));
      const bool partial = !(va && vb && kb >= kmin && kb + kStepKeys <= kmax);
      if (okw && partial) {
        // Keys of the step outside the run's range or on a missing page may
        // hold stale or uninitialised data: zero their value rows (this CTA's
        // columns) before P.V reads them.  Thread i of the group zeroes key row i.
        okw = __all_sync(0xffffffffu, mbar_wait(smem_addr(vfull + sv), (j / kStagesV) & 1, abort_flag));
        const int key = rl;
        const bool vpage = key < kPage ? va : vb;
        if (okw && (!vpage || kb + key < kmin || kb + key >= kmax)) {
          uint8_t* vrow = smem + L::vring + size_t(sv) * L::kVStage + (key >> 6) * kBoxBytes + (key & 63) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tc_fence_after();
      float x[kStepKeys];
      if (okw) {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(sc, r0);
        tmem_ld32(sc + 32, r1);
        tmem_ld32(sc + 64, r2);
        tmem_ld32(sc + 96, r3);
        tmem_ld_wait();
        // S_grp may take the next scores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(sfree0 + grp * 8);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(r0[i]);
          x[32 + i] = __uint_as_float(r1[i]);
          x[64 + i] = __uint_as_float(r2[i]);
          x[96 + i] = __uint_as_float(r3[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kStepKeys; ++i) x[i] = -INFINITY;
      }
      // visible keys of this step for this row: [a0, e0), minus a missing page
      const bool in_run = live && cur.run == run_id;
      const int ka = in_run ? max(lo - kb, 0) : kStepKeys;
      const int ke = in_run ? max(ka, min(hi - kb, kStepKeys)) : kStepKeys;
      const int ma = va ? 0 : kPage, me = vb ? kStepKeys : kPage;  // keys on valid pages: [ma, me)
      const int a0 = max(ka, ma), e0 = min(ke, me);
      if (!__all_sync(0xffffffffu, a0 == 0 && e0 == kStepKeys)) {
#pragma unroll
        for (int i = 0; i < kStepKeys; ++i) x[i] = (i >= a0 && i < e0) ? x[i] : -INFINITY;
      }
      // row max as a tree of independent three-input maxima
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        m8[k] = fmax3(x[k], x[8 + k], x[16 + k]);
#pragma unroll
        for (int i = 24; i < kStepKeys - 8; i += 16) m8[k] = fmax3(m8[k], x[i + k], x[i + 8 + k]);
        m8[k] = fmaxf(m8[k], x[kStepKeys - 8 + k]);
      }
      const float mraw = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      const float mx = mraw == -INFINITY ? -INFINITY : mraw * p.scale_log2;  // log2 units
      // the row's running max before this step, from the group of step j - 1
      if (j > 0) {
        named_barrier_sync(bar_sub, 64);
        m_ref = hand_m[((j - 1) & 1) * kRows + rl];
        okw = okw && hand_ok[((j - 1) & 1) * kRows + rl] != 0;
      }
      ok = __all_sync(0xffffffffu, okw);
      // new running max: it moves only when this step's max exceeds it by
      // more than 2^8, and then O is rescaled
      float m_new = m_ref, alpha = 1.f;
      if (mx != -INFINITY) {
        if (m_ref == -INFINITY) {
          m_new = mx;
        } else if (mx > m_ref + kRescaleLog2) {
          m_new = mx;
          alpha = exp2f(m_ref - mx);
        }
      }
      // hand it on before the exponentials, so the other group can go on
      if (j + 1 < nsteps) {
        hand_m[(j & 1) * kRows + rl] = m_new;
        hand_ok[(j & 1) * kRows + rl] = ok ? 1 : 0;
        __syncwarp();
        named_barrier_arrive(bar_pub, 64);
      }
      if (!ok) break;
      m_ref = m_new;
      // this group's partial sum follows the row's reference
      if (m_part != m_ref) {
        if (m_part != -INFINITY) l_part *= exp2f(m_part - m_ref);
        m_part = m_ref;
      }
      // probabilities 2^(s * scale * log2(e) - m_ref), packed to bf16 over
      // the first 64 columns of S_grp (paired fp32: one fma and one add per
      // two keys)
      const float nbase = m_ref == -INFINITY ? 0.f : -m_ref;
      const uint64_t c2 = f32x2(p.scale_log2, p.scale_log2), n2 = f32x2(nbase, nbase);
      // P_grp is free once P.V of step j - 2 has read it.  (This group waited
      // for P.V of step j - 4 before it wrote P at step j - 2, so pvdone[grp]
      // is at most one phase behind step j - 2 here, never two.)
      if (j >= 2) stuck = stuck || !__all_sync(0xffffffffu, mbar_wait(smem_addr(pvdone + grp), ((j - 2) >> 1) & 1, abort_flag));
      tc_fence_after();
      uint64_t s2[4] = {0ull, 0ull, 0ull, 0ull};  // running sums, two keys per register
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float a0v, a1v;
          f32x2_split(fma_f32x2(f32x2(x[hh * 32 + 2 * i], x[hh * 32 + 2 * i + 1]), c2, n2), a0v, a1v);
          const float e0v = ex2_approx(a0v), e1v = ex2_approx(a1v);
          s2[i & 3] = add_f32x2(s2[i & 3], f32x2(e0v, e1v));
          pk[i] = pack_bf16x2(e0v, e1v);
        }
        tmem_st16(pcol + hh * 16, pk);
      }
      if (__any_sync(0xffffffffu, alpha != 1.f) && j >= 1) {
        // the running max grew: rescale this row of O once P.V of step j - 1
        // (written by the other group) has finished, before P.V of step j.
        // (P.V runs in step order and the wait above saw step j - 2 finish,
        // so step j - 3 has finished too: that barrier is at most one phase
        // behind step j - 1.)
        // (this group's hand-off for step j + 1 has gone out already: if the
        // wait gives up, the failure travels with its next hand-off instead)
        stuck = stuck || !__all_sync(0xffffffffu, mbar_wait(smem_addr(pvdone + ((j - 1) & 1)), ((j - 1) >> 1) & 1,
                                                             abort_flag));
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < (stuck ? 0 : L::kPvN / 32); ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lanes + L::kColO + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tmem + lanes + L::kColO + c * 32, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (partial) mbar_arrive_cluster(pfull0 + grp * 8);  // publishes the zeroed value rows
        else mbar_arrive_remote(pfull0 + grp * 8);
      }
      {
        float u0, u1;
        f32x2_split(add_f32x2(add_f32x2(s2[0], s2[1]), add_f32x2(s2[2], s2[3])), u0, u1);
        l_part += u0 + u1;
      }
    }
    // ---- normalise and store this row: group g stores half g of head_dim ----
    // (the last P.V commits to a barrier of its own: here pvdone may be one
    // phase short of it or already past it, which a parity wait cannot tell)
    if (nsteps > 0) {
      const bool okw = ok && !stuck && __all_sync(0xffffffffu, mbar_wait(smem_addr(odone), 0, abort_flag));
      tc_fence_after();
      fin_m[grp * kRows + rl] = m_part;
      fin_l[grp * kRows + rl] = l_part;
      fin_ok[grp * kRows + rl] = okw ? 1 : 0;
      named_barrier_sync(bar_fin, 64);
      const float mo = fin_m[(grp ^ 1) * kRows + rl], lo_ = fin_l[(grp ^ 1) * kRows + rl];
      ok = __all_sync(0xffffffffu, okw && fin_ok[(grp ^ 1) * kRows + rl] != 0);
      // both partial sums relative to the final reference (the larger one)
      const float mf = fmaxf(m_part, mo);
      const float la = m_part == -INFINITY ? 0.f : l_part * exp2f(m_part - mf);
      const float lb = mo == -INFINITY ? 0.f : lo_ * exp2f(mo - mf);
      l_part = grp == 0 ? la + lb : lb + la;
    }
    // this group's half of the row: all of its columns read from tensor
    // memory at once, then stored 16 bytes at a time
    uint16_t* dst = p.out + qrow + grp * (D / 2);
    const float inv = l_part > 0.f ? 1.f / l_part : 0.f;
    uint32_t r[D / 2];
    if (ok && nsteps > 0) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t (&rc)[16] = *reinterpret_cast<uint32_t(*)[16]>(r + c * 16);
        tmem_ld16(tmem + lanes + L::kColO + grp * (D / 2) + c * 16, rc);
      }
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < D / 2; ++i) r[i] = 0u;
    }
    if (tl < nt) {
      uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = live ? __uint_as_float(r[8 * i + k]) * inv : 0.f;
        o[i] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                          pack_bf16x2(v[6], v[7]));
      }
    }
  }
  if (*abort_flag && lane == 0 && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
  // neither CTA frees its tensor memory or leaves while the pair's products,
  // copies or remote arrivals may still touch it
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem2_dealloc(tmem, L::kTmemCols);
}

template <int D>
cudaError_t launch_chunk_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const ChunkParams& p,
                           cudaStream_t stream) {
  const int bytes = static_cast<int>(TcSmem<D>::bytes);
  cudaError_t err = set_max_dynamic_smem(reinterpret_cast<const void*>(chunk_kernel<D>), bytes);
  if (err != cudaSuccess) return err;
  const long long grid = 2ll * p.num_tiles * p.hkv;  // a cluster of two CTAs per (tile, kv head)
  if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
  chunk_kernel<D><<<static_cast<unsigned>(grid), kThreads, bytes, stream>>>(kmap, vmap, p);
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
