// K4: packed prompt chunks (prefill_paged / the prompt part of step_paged).
//
// Every chunk token attends over its own row's pages up to its position (and
// the window).  A CTA takes one tile of consecutive pack tokens and one kv
// head: tile_tokens = 128 / G tokens times the G query heads of that kv head
// gives 128 query rows, 16 per consumer warp (row m = token * G + head).
// Tokens of a tile are grouped into runs of equal table rows; for each run
// the producer warp streams the row's pages covering the run's key range
// through a ring of TMA stages (128-byte swizzle), and the eight consumer
// warps run the FlashAttention recurrence per page:
//   S[16 rows, 64 keys]  = Q K^T   (mma m16n8k16, K^T fragments via ldmatrix)
//   O[16 rows, D]       += P V     (P reused from the S accumulators,
//                                   V fragments via ldmatrix.trans)
// with a per-row mask: same run, lo <= key <= position.
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

constexpr int kWarps = 8;                  // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kRows = kWarps * 16;         // query rows per tile

struct ChunkStage {
  int run, key_base, valid;
};

template <int D>
struct ChunkSmem {
  static constexpr int NB = boxes_for(D);
  static constexpr int kStageBytes = 2 * NB * kBoxBytes;
  static constexpr size_t stages = 0;
  static constexpr size_t bars = stages + size_t(kStages) * kStageBytes;
  static constexpr size_t info = bars + (2 * kStages + 1) * sizeof(uint64_t);
  static constexpr size_t tok = info + kStages * sizeof(ChunkStage);
  static constexpr size_t runs = tok + 3 * kRows * 4;     // token lo, hi (exclusive), run
  static constexpr size_t misc = runs + 4 * kRows * 4;    // run row, kmin, kmax, pages
  static constexpr size_t bytes = misc + 64 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const ChunkParams p) {
  using L = ChunkSmem<D>;
  constexpr int NB = L::NB;
  constexpr int DK = D / 16;   // k-steps of Q K^T
  constexpr int DN = D / 8;    // n-tiles of the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* zero_bar = empty_bar + kStages;  // consumers finished zeroing a partial page
  ChunkStage* info = reinterpret_cast<ChunkStage*>(smem + L::info);
  int* tok_lo = reinterpret_cast<int*>(smem + L::tok);
  int* tok_hi = tok_lo + kRows;
  int* tok_run = tok_hi + kRows;
  int* run_row = reinterpret_cast<int*>(smem + L::runs);
  int* run_kmin = run_row + kRows;
  int* run_kmax = run_kmin + kRows;
  int* run_pages = run_kmax + kRows;
  int* misc = reinterpret_cast<int*>(smem + L::misc);  // [0] runs, [1] stages, [2] abort
  volatile int* abort_flag = misc + 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.group;
  const int TQ = p.tile_tokens;
  const int tile = p.num_tiles - 1 - static_cast<int>(blockIdx.x);  // later tokens first
  const int h = blockIdx.y;
  const int t0 = tile * TQ;
  const int nt = min(TQ, p.P - t0);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(full_bar + s), 1);
      mbar_init(smem_addr(empty_bar + s), kWarps);
    }
    mbar_init(smem_addr(zero_bar), kWarps * 32);
    misc[2] = 0;
    fence_mbarrier_init();
  }
  // ---- tokens of the tile ----
  if (tid < TQ) {
    int lo = 0, hi = 0, bad = 0;
    if (tid < nt) {
      const int t = t0 + tid;
      const int pos = p.positions[t];
      const int row = p.rows[t];
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
    if (bad && h == 0 && p.status != nullptr) atomicOr(p.status, bad);
  }
  __syncthreads();
  if (tid == 0) {
    int nr = 0, cur = -1, stages = 0;
    for (int i = 0; i < nt; ++i) {
      if (tok_hi[i] <= tok_lo[i]) {
        tok_run[i] = -1;
        continue;
      }
      const int row = p.rows[t0 + i];
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
      stages += run_pages[r];
    }
    misc[0] = nr;
    misc[1] = stages;
  }
  __syncthreads();
  const int nruns = misc[0];
  const int nstages = misc[1];

  if (warp == kWarps) {
    // ============================== producer ==============================
    if (lane != 0) return;
    tma_prefetch_descriptor(&kmap);
    tma_prefetch_descriptor(&vmap);
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
        ChunkStage si{run, lp * kPage, 1};
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
    const int issued = k;
    for (int kk = max(0, issued - kStages); kk < issued; ++kk) {
      const uint32_t fb = smem_addr(full_bar + kk % kStages);
      const uint64_t t_0 = global_timer_ns();
      while (!mbar_try_wait(fb, (kk / kStages) & 1) && global_timer_ns() - t_0 < kWaitLimitNs) {
      }
    }
    if (*abort_flag && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
    return;
  }

  // ============================== consumers ==============================
  const int c = lane & 3;
  const int r = lane >> 2;
  const int m0 = warp * 16 + r, m1 = m0 + 8;
  const int tk0 = m0 / G, g0 = m0 % G;
  const int tk1 = m1 / G, g1 = m1 % G;
  const int lo0 = tok_lo[tk0], hi0 = tok_hi[tk0], run0 = tok_run[tk0];
  const int lo1 = tok_lo[tk1], hi1 = tok_hi[tk1], run1 = tok_run[tk1];

  // Q fragments (A operand, rows m0 / m1)
  uint32_t qa[DK][4];
  {
    const uint16_t* q0 = p.q + (static_cast<size_t>(t0 + tk0) * p.hq + static_cast<size_t>(h) * G + g0) * D;
    const uint16_t* q1 = p.q + (static_cast<size_t>(t0 + tk1) * p.hq + static_cast<size_t>(h) * G + g1) * D;
    const bool ok0 = run0 >= 0, ok1 = run1 >= 0;
#pragma unroll
    for (int kk = 0; kk < DK; ++kk) {
      const int e = kk * 16 + 2 * c;
      qa[kk][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + e) : 0u;
      qa[kk][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + e) : 0u;
      qa[kk][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + e + 8) : 0u;
      qa[kk][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + e + 8) : 0u;
    }
  }
  float o[DN][4];
#pragma unroll
  for (int n = 0; n < DN; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_0 = -INFINITY, m_1 = -INFINITY, l_0 = 0.f, l_1 = 0.f;
  uint32_t zero_phase = 0;

  for (int k = 0; k < nstages; ++k) {
    const int s = k % kStages;
    if (!mbar_wait(smem_addr(full_bar + s), (k / kStages) & 1, abort_flag)) break;
    const ChunkStage si = info[s];
    const uint8_t* kbuf = smem + L::stages + size_t(s) * L::kStageBytes;
    const uint8_t* vbuf = kbuf + NB * kBoxBytes;
    const int kb = si.key_base;
    if (si.valid) {
      const int kmin = run_kmin[si.run], kmax = run_kmax[si.run];
      if (kb < kmin || kb + kPage > kmax) {
        // Keys of this page outside the run's range may hold stale or
        // uninitialised data: zero their value rows before anyone reads them.
        uint8_t* vw = const_cast<uint8_t*>(vbuf);
        for (int i = tid; i < kPage * NB * 8; i += kWarps * 32) {
          const int key = i / (NB * 8);
          const int rest = i % (NB * 8);
          if (kb + key < kmin || kb + key >= kmax)
            *reinterpret_cast<uint4*>(vw + (rest >> 3) * kBoxBytes + key * 128 + (rest & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_addr(zero_bar));
        if (!mbar_wait(smem_addr(zero_bar), zero_phase & 1, abort_flag)) break;
        ++zero_phase;
      }
    }
    // does any row of this warp see a key of this page?
    const bool in0 = run0 == si.run && lo0 < kb + kPage && hi0 > kb;
    const bool in1 = run1 == si.run && lo1 < kb + kPage && hi1 > kb;
    if (si.valid && __any_sync(0xffffffffu, in0 || in1)) {
      const uint32_t kaddr = smem_addr(kbuf);
      const uint32_t vaddr = smem_addr(vbuf);
      float sc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DK; ++kk) {
#pragma unroll
        for (int nn = 0; nn < 4; ++nn) {
          const int key = nn * 16 + (lane & 7) + (lane >> 4) * 8;
          const int chunk = kk * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kaddr + (chunk >> 3) * kBoxBytes + swz128(key, chunk & 7), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * nn], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma_bf16_16816(sc[2 * nn + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
      // mask + row maxima
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int key = kb + n * 8 + 2 * c;
        const bool a0 = in0 && key >= lo0 && key < hi0;
        const bool a1 = in0 && key + 1 >= lo0 && key + 1 < hi0;
        const bool b0 = in1 && key >= lo1 && key < hi1;
        const bool b1 = in1 && key + 1 >= lo1 && key + 1 < hi1;
        sc[n][0] = a0 ? sc[n][0] * p.scale_log2 : -INFINITY;
        sc[n][1] = a1 ? sc[n][1] * p.scale_log2 : -INFINITY;
        sc[n][2] = b0 ? sc[n][2] * p.scale_log2 : -INFINITY;
        sc[n][3] = b1 ? sc[n][3] * p.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m_0, mx0), mn1 = fmaxf(m_1, mx1);
      const float base0 = mn0 == -INFINITY ? 0.f : mn0;
      const float base1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m_0 - base0), al1 = exp2f(m_1 - base1);
      m_0 = mn0;
      m_1 = mn1;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pa[4][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float e0 = exp2f(sc[n][0] - base0), e1 = exp2f(sc[n][1] - base0);
        const float e2 = exp2f(sc[n][2] - base1), e3 = exp2f(sc[n][3] - base1);
        rs0 += e0 + e1;
        rs1 += e2 + e3;
        // A fragment of P for k-step n / 2: n even -> regs 0, 1; n odd -> regs 2, 3
        pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16x2(e0, e1);
        pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(e2, e3);
      }
      l_0 = l_0 * al0 + rs0;
      l_1 = l_1 * al1 + rs1;
#pragma unroll
      for (int n = 0; n < DN; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int nd = 0; nd < DN / 2; ++nd) {
          const int key = j * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int chunk = nd * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(vaddr + (chunk >> 3) * kBoxBytes + swz128(key, chunk & 7), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * nd], pa[j][0], pa[j][1], pa[j][2], pa[j][3], b0, b1);
          mma_bf16_16816(o[2 * nd + 1], pa[j][0], pa[j][1], pa[j][2], pa[j][3], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(empty_bar + s));
  }
  if (*abort_flag) {
    if (lane == 0 && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
  }

  // ---- normalise and store ----
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_0 += __shfl_xor_sync(0xffffffffu, l_0, off);
    l_1 += __shfl_xor_sync(0xffffffffu, l_1, off);
  }
  const float inv0 = l_0 > 0.f ? 1.f / l_0 : 0.f;
  const float inv1 = l_1 > 0.f ? 1.f / l_1 : 0.f;
  if (tk0 < nt) {
    uint16_t* dst = p.out + (static_cast<size_t>(t0 + tk0) * p.hq + static_cast<size_t>(h) * G + g0) * D;
#pragma unroll
    for (int n = 0; n < DN; ++n)
      *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * c) = pack_bf16x2(o[n][0] * inv0, o[n][1] * inv0);
  }
  if (tk1 < nt) {
    uint16_t* dst = p.out + (static_cast<size_t>(t0 + tk1) * p.hq + static_cast<size_t>(h) * G + g1) * D;
#pragma unroll
    for (int n = 0; n < DN; ++n)
      *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * c) = pack_bf16x2(o[n][2] * inv1, o[n][3] * inv1);
  }
}

template <int D>
cudaError_t launch_chunk_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const ChunkParams& p,
                           cudaStream_t stream) {
  const int bytes = static_cast<int>(ChunkSmem<D>::bytes);
  cudaError_t err =
      cudaFuncSetAttribute(chunk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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

cudaError_t launch_chunk(const CUtensorMap& kmap, const CUtensorMap& vmap, const ChunkParams& p,
                         int head_dim, cudaStream_t stream) {
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
