// K2 + K3: paged split-KV decode attention and its log-sum-exp combine.
//
// Work decomposition.  Decode row b at position p sees keys
// [max(0, p - window + 1), p], i.e. np_b pages of 64 (the first and last may
// be partial).  Each (row, kv head) pair is a run of np_b page-heads; the runs
// of all pairs, (b, h) with h fastest, are laid end to end and the resulting
// stream of page-heads is cut into gridDim.x equal pieces, one per persistent
// CTA.  A pair that falls inside one CTA is finished there (output written
// directly); a pair cut by CTA boundaries leaves one partial result per CTA
// (unnormalised output, running max, running sum) and the combine kernel
// merges them.  Pair q = b * Hkv + h touching CTA c writes segment q + c,
// which is unique because consecutive pairs never go back to an earlier CTA.
//
// CTA structure (160 threads).  Warp 4 is the producer: one lane walks the
// CTA's page-heads, reads the page table, and loads each page's K and V
// (64 positions x head_dim bf16, contiguous in the head-major pool) with 2-D
// TMA tile copies into a ring of shared-memory stages (128-byte swizzle),
// completing on the stage's "full" mbarrier.  Warps 0-3 consume every stage:
// warp w owns keys 16w .. 16w + 15 of the page and keeps its own online
// softmax state.  Per page and warp:
//   S^T[16 keys, 8 heads] = K[16 keys, D] * Q^T  (mma m16n8k16, keys as M,
//                                                  the GQA group padded to N = 8)
//   O^T[D, 8 heads]      += V^T[D, 16 keys] * P^T (V^T via ldmatrix.trans,
//                                                  P^T via movmatrix.trans of
//                                                  the S fragment)
// At the end of a pair's run inside the CTA the four warps merge through
// shared memory.
//
// Sources: "Phi-3 Mini 4K Instruct -- files", src/attention.linnet
// (decode_rows: a row attends over itself up to its position; window_mask;
// scale rsqrt(head_dim)); "Mistral 7B Instruct v0.3", Entries table
// (decode_paged: the pool, pages of 64, table[b]).
#include <cfloat>

#include "common.cuh"
#include "ptx.cuh"

namespace lnk {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kPairFirst = 1;
constexpr int kPairLast = 2;
constexpr int kPairWhole = 4;

struct StageInfo {
  int b, h, klo, khi, flags, seg;
};

template <int D>
struct DecodeSmem {
  static constexpr int NB = boxes_for(D);
  static constexpr int kStageBytes = 2 * NB * kBoxBytes;          // K boxes, then V boxes
  static constexpr int kOStride = D + 4;                          // padded staging row
  static constexpr size_t stages = 0;
  static constexpr size_t bars = stages + size_t(kStages) * kStageBytes;
  static constexpr size_t info = bars + (2 * kStages + 2) * sizeof(uint64_t);
  static constexpr size_t ostage = info + kStages * sizeof(StageInfo);
  static constexpr size_t mstage = ostage + size_t(kConsumerWarps) * kMaxGroup * kOStride * 4;
  static constexpr size_t lstage = mstage + kConsumerWarps * kMaxGroup * 4;
  static constexpr size_t misc = lstage + kConsumerWarps * kMaxGroup * 4;  // abort flag, totals
  static constexpr size_t pref = misc + 64;
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  using L = DecodeSmem<D>;
  constexpr int NB = L::NB;
  constexpr int DK = D / 16;  // k-steps of Q.K and d-tiles of P.V
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* merge_bar = empty_bar + kStages;  // [0]: staging written, [1]: staging read
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + L::info);
  float* ost = reinterpret_cast<float*>(smem + L::ostage);
  float* mst = reinterpret_cast<float*>(smem + L::mstage);
  float* lst = reinterpret_cast<float*>(smem + L::lstage);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc);
  int* scan_tot = reinterpret_cast<int*>(smem + L::ostage);  // reuses the staging area at start
  int* pref = reinterpret_cast<int*>(smem + L::pref);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int B = p.B;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(full_bar + s), 1);
      mbar_init(smem_addr(empty_bar + s), kConsumerWarps);
    }
    mbar_init(smem_addr(merge_bar + 0), kConsumerWarps * 32);
    mbar_init(smem_addr(merge_bar + 1), kConsumerWarps * 32);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_descriptor(&kmap);
    tma_prefetch_descriptor(&vmap);
  }

  // ---- per-row visible page counts and their prefix sums (all threads) ----
  {
    const int chunk = (B + kThreads - 1) / kThreads;
    const int r0 = min(B, tid * chunk), r1 = min(B, r0 + chunk);
    int bad = 0, run = 0;
    for (int b = r0; b < r1; ++b) {
      run += visible_pages(p.positions[b], p.window, p.pages_per_row, &bad);
      pref[b + 1] = run;
    }
    if (bad && p.status != nullptr && blockIdx.x == 0) atomicOr(p.status, bad);
    scan_tot[tid] = run;
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int i = 0; i < kThreads; ++i) {
        const int v = scan_tot[i];
        scan_tot[i] = acc;
        acc += v;
      }
      pref[0] = 0;
    }
    __syncthreads();
    const int off = scan_tot[tid];
    for (int b = r0; b < r1; ++b) pref[b + 1] += off;
    __syncthreads();
  }

  const long long total = static_cast<long long>(pref[B]) * p.hkv;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long start = min(total, static_cast<long long>(blockIdx.x) * per);
  const long long end = min(total, start + per);
  if (blockIdx.x == 0) {
    if (tid == 0) p.ws_meta[0] = static_cast<int>(per);
    for (int b = tid; b <= B; b += kThreads) p.ws_pref[b] = pref[b];
  }
  if (start >= end) return;

  if (warp == kConsumerWarps) {
    // ============================== producer ==============================
    if (lane != 0) return;
    // locate the pair holding page-head `start`
    int lo_b = 0, hi_b = B - 1;  // largest b with hkv * pref[b] <= start
    while (lo_b < hi_b) {
      const int mid = (lo_b + hi_b + 1) >> 1;
      if (static_cast<long long>(pref[mid]) * p.hkv <= start) lo_b = mid; else hi_b = mid - 1;
    }
    int b = lo_b;
    int np = pref[b + 1] - pref[b];
    long long rem = start - static_cast<long long>(pref[b]) * p.hkv;
    int h = static_cast<int>(rem / np);
    int j = static_cast<int>(rem % np);
    int pos = p.positions[b];
    int lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
    int first_page = lo / kPage;
    const int* trow = p.table + static_cast<long long>(b) * p.pages_per_row;

    int k = 0;
    for (long long gi = start; gi < end; ++gi, ++k) {
      const int s = k % kStages;
      if (k >= kStages) {
        if (!mbar_wait(smem_addr(empty_bar + s), ((k / kStages) - 1) & 1, abort_flag)) break;
      }
      const int lp = first_page + j;
      const int page = trow[lp];
      StageInfo si;
      si.b = b;
      si.h = h;
      si.klo = max(lo - lp * kPage, 0);
      si.khi = min(pos - lp * kPage + 1, kPage);
      const long long pair_start = gi - j;
      si.flags = ((gi == start || j == 0) ? kPairFirst : 0) | ((gi == end - 1 || j == np - 1) ? kPairLast : 0) |
                 ((pair_start >= start && pair_start + np <= end) ? kPairWhole : 0);
      si.seg = b * p.hkv + h + static_cast<int>(blockIdx.x);
      const uint32_t fb = smem_addr(full_bar + s);
      if (page < 0 || page >= p.num_pages) {
        if (p.status != nullptr) atomicOr(p.status, LNK_DEV_BAD_PAGE);
        si.klo = si.khi = 0;
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
      // advance to the next page-head
      if (++j == np) {
        j = 0;
        if (++h == p.hkv) {
          h = 0;
          do { ++b; } while (b < B && pref[b + 1] == pref[b]);
          if (b < B) {
            np = pref[b + 1] - pref[b];
            pos = p.positions[b];
            lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
            first_page = lo / kPage;
            trow = p.table + static_cast<long long>(b) * p.pages_per_row;
          }
        }
      }
    }
    // Drain: do not leave the CTA while a copy may still land in its memory.
    const int issued = k;
    for (int kk = max(0, issued - kStages); kk < issued; ++kk) {
      const int s = kk % kStages;
      const uint32_t fb = smem_addr(full_bar + s);
      if (!mbar_try_wait(fb, (kk / kStages) & 1)) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(fb, (kk / kStages) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    if (*abort_flag && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
    return;
  }

  // ============================== consumers ==============================
  const int c = lane & 3;    // column pair: heads 2c, 2c + 1
  const int r = lane >> 2;   // row within an 8-row group
  const int key0 = warp * 16;
  const uint8_t* stage_base = smem + L::stages;

  uint32_t qf[DK][2];
  float o[DK][4];
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  uint32_t merges = 0;

  const int nsteps = static_cast<int>(end - start);
  for (int k = 0; k < nsteps; ++k) {
    const int s = k % kStages;
    if (!mbar_wait(smem_addr(full_bar + s), (k / kStages) & 1, abort_flag)) break;
    const StageInfo si = info[s];
    if (si.flags & kPairFirst) {
      const uint16_t* qrow = p.q + (static_cast<size_t>(si.b) * p.hq + static_cast<size_t>(si.h) * p.group) * D;
      const bool gv = r < p.group;
#pragma unroll
      for (int kk = 0; kk < DK; ++kk) {
        qf[kk][0] = gv ? *reinterpret_cast<const uint32_t*>(qrow + r * D + kk * 16 + 2 * c) : 0u;
        qf[kk][1] = gv ? *reinterpret_cast<const uint32_t*>(qrow + r * D + kk * 16 + 8 + 2 * c) : 0u;
      }
#pragma unroll
      for (int dt = 0; dt < DK; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
      m_a = m_b = -INFINITY;
      l_a = l_b = 0.f;
    }
    if (si.khi > si.klo && si.klo < key0 + 16 && si.khi > key0) {
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
      // ---- S^T = K Q^T ----
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int key = key0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < DK; ++kk) {
          const int chunk = kk * 2 + (lane >> 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kaddr + (chunk >> 3) * kBoxBytes + swz128(key, chunk & 7), a0, a1, a2, a3);
          mma_bf16_16816(sc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
      }
      // ---- mask, online softmax (log2 domain) ----
      const int kr0 = key0 + r, kr1 = kr0 + 8;
      const bool v0 = kr0 >= si.klo && kr0 < si.khi;
      const bool v1 = kr1 >= si.klo && kr1 < si.khi;
      const float s0 = v0 ? sc[0] * p.scale_log2 : -INFINITY;
      const float s1 = v0 ? sc[1] * p.scale_log2 : -INFINITY;
      const float s2 = v1 ? sc[2] * p.scale_log2 : -INFINITY;
      const float s3 = v1 ? sc[3] * p.scale_log2 : -INFINITY;
      float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
      }
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
      const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
      const float al_a = exp2f(m_a - base_a), al_b = exp2f(m_b - base_b);
      const float p0 = exp2f(s0 - base_a), p1 = exp2f(s1 - base_b);
      const float p2 = exp2f(s2 - base_a), p3 = exp2f(s3 - base_b);
      l_a = l_a * al_a + (p0 + p2);
      l_b = l_b * al_b + (p1 + p3);
      m_a = mn_a;
      m_b = mn_b;
#pragma unroll
      for (int dt = 0; dt < DK; ++dt) {
        o[dt][0] *= al_a;
        o[dt][1] *= al_b;
        o[dt][2] *= al_a;
        o[dt][3] *= al_b;
      }
      // ---- O^T += V^T P^T ----
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
      {
        const int key = key0 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int dt = 0; dt < DK; ++dt) {
          const int chunk = dt * 2 + ((lane >> 3) & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(vaddr + (chunk >> 3) * kBoxBytes + swz128(key, chunk & 7), a0, a1, a2, a3);
          mma_bf16_16816(o[dt], a0, a1, a2, a3, pb0, pb1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(empty_bar + s));

    if (si.flags & kPairLast) {
      // ---- merge the four warps' states for this pair ----
      float la = l_a, lb = l_b;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, off);
        lb += __shfl_xor_sync(0xffffffffu, lb, off);
      }
      if (lane < 4) {
        mst[warp * kMaxGroup + 2 * c] = m_a;
        mst[warp * kMaxGroup + 2 * c + 1] = m_b;
        lst[warp * kMaxGroup + 2 * c] = la;
        lst[warp * kMaxGroup + 2 * c + 1] = lb;
      }
      float* ow = ost + size_t(warp) * kMaxGroup * L::kOStride;
#pragma unroll
      for (int dt = 0; dt < DK; ++dt) {
        ow[(2 * c) * L::kOStride + dt * 16 + r] = o[dt][0];
        ow[(2 * c + 1) * L::kOStride + dt * 16 + r] = o[dt][1];
        ow[(2 * c) * L::kOStride + dt * 16 + r + 8] = o[dt][2];
        ow[(2 * c + 1) * L::kOStride + dt * 16 + r + 8] = o[dt][3];
      }
      mbar_arrive(smem_addr(merge_bar + 0));
      if (!mbar_wait(smem_addr(merge_bar + 0), merges & 1, abort_flag)) break;
      const int G = p.group;
      const bool whole = (si.flags & kPairWhole) != 0;
      for (int idx = tid; idx < G * D; idx += kConsumerWarps * 32) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mst[w * kMaxGroup + g]);
        float Lsum = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = mst[w * kMaxGroup + g];
            if (mw != -INFINITY) {
              const float f = exp2f(mw - M);
              Lsum += lst[w * kMaxGroup + g] * f;
              acc += ost[(size_t(w) * kMaxGroup + g) * L::kOStride + d] * f;
            }
          }
        }
        if (whole) {
          const float val = Lsum > 0.f ? acc / Lsum : 0.f;
          p.out[(static_cast<size_t>(si.b) * p.hq + static_cast<size_t>(si.h) * G + g) * D + d] =
              __bfloat16_as_ushort(__float2bfloat16_rn(val));
        } else {
          p.ws_o[(static_cast<size_t>(si.seg) * G + g) * D + d] = acc;
          if (d == 0) {
            p.ws_ml[(static_cast<size_t>(si.seg) * G + g) * 2 + 0] = M;
            p.ws_ml[(static_cast<size_t>(si.seg) * G + g) * 2 + 1] = Lsum;
          }
        }
      }
      mbar_arrive(smem_addr(merge_bar + 1));
      if (!mbar_wait(smem_addr(merge_bar + 1), merges & 1, abort_flag)) break;
      ++merges;
    }
  }
  if (*abort_flag && lane == 0 && p.status != nullptr) atomicOr(p.status, LNK_DEV_TIMEOUT);
}

// Merges the partial results of (row, kv head) pairs that were cut by CTA
// boundaries, and zeroes the outputs of rows with no visible keys.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p) {
  const int q = blockIdx.x;
  const int b = q / p.hkv, h = q % p.hkv;
  const int G = p.group;
  const int np = p.ws_pref[b + 1] - p.ws_pref[b];
  uint16_t* out = p.out + (static_cast<size_t>(b) * p.hq + static_cast<size_t>(h) * G) * D;
  if (np == 0) {
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) out[idx] = 0;
    return;
  }
  const long long per = p.ws_meta[0];
  const long long start = static_cast<long long>(p.ws_pref[b]) * p.hkv + static_cast<long long>(h) * np;
  const long long end = start + np;
  const int c0 = static_cast<int>(start / per), c1 = static_cast<int>((end - 1) / per);
  if (c0 == c1) return;  // finished inside one CTA
  const int seg0 = q + c0, nseg = c1 - c0 + 1;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, d = idx % D;
    float M = -INFINITY;
    for (int s = 0; s < nseg; ++s) M = fmaxf(M, p.ws_ml[(static_cast<size_t>(seg0 + s) * G + g) * 2]);
    float Lsum = 0.f, acc = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < nseg; ++s) {
        const size_t si = static_cast<size_t>(seg0 + s) * G + g;
        const float ms = p.ws_ml[si * 2];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - M);
        Lsum += p.ws_ml[si * 2 + 1] * f;
        acc += p.ws_o[si * D + d] * f;
      }
    }
    out[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(Lsum > 0.f ? acc / Lsum : 0.f));
  }
}

template <int D>
cudaError_t launch_decode_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                            const DecodeLaunch& launch, cudaStream_t stream) {
  decode_kernel<D><<<launch.grid, kThreads, launch.smem_bytes, stream>>>(kmap, vmap, p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  combine_kernel<D><<<p.B * p.hkv, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t prepare_t(int B, DecodeLaunch* launch) {
  const size_t bytes = DecodeSmem<D>::bytes(B);
  cudaError_t err = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
  if (err != cudaSuccess) return err;
  launch->smem_bytes = static_cast<int>(bytes);
  launch->grid = device_sm_count();
  return cudaSuccess;
}

}  // namespace

DecodeWorkspace decode_workspace_layout(int rows, int hkv, int group, int head_dim, int grid) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  DecodeWorkspace w;
  const size_t segs = static_cast<size_t>(rows) * hkv + static_cast<size_t>(grid);
  w.meta = 0;
  w.pref = up(w.meta + 64);
  w.ml = up(w.pref + (static_cast<size_t>(rows) + 1) * 4);
  w.o = up(w.ml + segs * group * 2 * 4);
  w.total = up(w.o + segs * group * static_cast<size_t>(head_dim) * 4);
  return w;
}

cudaError_t decode_prepare(int head_dim, int B, DecodeLaunch* launch) {
  switch (head_dim) {
    case 64: return prepare_t<64>(B, launch);
    case 96: return prepare_t<96>(B, launch);
    case 128: return prepare_t<128>(B, launch);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                          int head_dim, const DecodeLaunch& launch, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch_decode_t<64>(kmap, vmap, p, launch, stream);
    case 96: return launch_decode_t<96>(kmap, vmap, p, launch, stream);
    case 128: return launch_decode_t<128>(kmap, vmap, p, launch, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lnk
