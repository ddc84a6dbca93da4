// LM-head GEMM fused with the vocab-parallel cross-entropy statistics: the
// logits z = X W_i^T of every vocabulary shard are formed tile by tile on the
// tensor cores and reduced to per-row (max, sum of exponentials) partials and
// the target logit in the tile's epilogue, so the [s, V] logits are never
// written.  This is the pages' "do not assemble the big tensor, move the
// later computation to where the data is" ("Distributed Training III: Model
// Parallelism", CMU 11-868 Lecture 16 notes, §5.5), applied one step earlier
// than the sharded loss: the LM head is [V, h] split along V ("LLM Internals"
// §7.3.4: [128256, 8192], 16032 rows per card at t = 8).
//
// Kernel shape (sm_100 family, one CTA per SM, persistent).  A CTA's tile is
// a pair of 128-row M tiles against one 256-column N tile, so each W tile
// brought into shared memory feeds two MMAs: 64 KB of operands per 64-deep
// K step instead of 48 KB per half the work, which is what kept the tensor
// pipe at 80 % with one M tile per CTA (shared memory fill, not L2, was the
// limit).
//   warp 0      one lane issues the TMA loads: two 128 x 64 tiles of X and a
//               256 x 64 tile of W_i per K step, 128-byte swizzled, into a
//               3-stage shared-memory ring (mbarrier full / empty);
//   warp 1      allocates 512 TMEM columns (the pair's two 128 x 256 fp32
//               accumulators); one lane issues tcgen05.mma (kind::f16, bf16
//               in, fp32 accumulate, M = 128, N = 256, K = 16 per
//               instruction), two per K slice, and commits each stage back to
//               the loader and each finished pair of accumulators to the
//               epilogue;
//   warps 2..5  the epilogue: each thread owns one row of each M tile (one
//               TMEM lane), reads the row's 256 fp32 values with tcgen05.ld,
//               masks the columns past the shard's end, folds them into a
//               running (max, sum exp) and picks up the target logit when
//               the row's target column falls in the tile.  With all 512
//               columns holding the pair, the next tile's MMAs wait for it
//               (a few percent of a tile's MMA time).
// CTA c takes M-tile pair (wave * gm + c % gm) and, in each wave, one of gn
// ranges of N tiles, the same for the gm CTAs of group c / gm: they read the
// same W tile at the same time (L2 hits), and the gn CTAs of a pair read the
// same X tiles.  A group's range moves on by one each wave, which spreads
// the longer ranges evenly over the groups.  Each CTA writes one partial per
// row for its range; the combine kernel of the sharded loss folds them in
// range order, i.e. in vocabulary order.
#include <cstring>

#include "vpce_kernels.cuh"
#include "vpce_tc.cuh"

namespace vpce {

namespace {

constexpr int kBM = 128;   // rows (tokens) per tile
constexpr int kBN = 256;   // vocabulary columns per tile
constexpr int kBK = 64;    // K elements per stage (one 128-byte swizzle atom of bf16)
constexpr int kUK = 16;    // K per tcgen05.mma for 16-bit inputs
constexpr int kMT = 2;     // M tiles per CTA tile (they share each W tile)
constexpr int kGStages = 3;
constexpr int kATile = kBM * kBK * 2;  // 16 KB
constexpr int kBTile = kBN * kBK * 2;  // 32 KB
constexpr int kGStage = kMT * kATile + kBTile;
constexpr int kGThreads = 192;  // 6 warps
constexpr int kTmemCols = 512;  // the pair's two accumulators of kBN fp32 columns
static_assert(kMT * kBN <= kTmemCols, "the pair's accumulators fit in TMEM");
constexpr int kMaxGemmShards = 32;
constexpr int kMaxGroupsPerWave = 16;  // M tiles that share a W tile (kMaxGroupsPerWave / kMT pairs)

struct GemmSmem {
  unsigned char stage[kGStages][kGStage];  // 1024-byte aligned (swizzle atoms): A0, A1, B
  uint64_t full[kGStages];
  uint64_t empty[kGStages];
  uint64_t acc_full;   // the pair's accumulators are complete
  uint64_t acc_empty;  // the epilogue has read them
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct GemmParams {
  CUtensorMap tmx;                  // X [s, h] bf16, box 64 x 128
  CUtensorMap tmw[kMaxGemmShards];  // W_i [w_i, h] bf16, box 64 x 256
  int t;
  int s;
  int k_steps;                      // h / 64
  int m_tiles, n_tiles, gm, gn;     // gm: M-tile pairs per wave
  int m_pairs;
  int vstart[kMaxGemmShards + 1];   // global column of each shard's first row
  int nstart[kMaxGemmShards + 1];   // first N tile of each shard
  const long long* targets;
  long long ignore_index;
  float2* part;                     // [gn][s]: (max, sum exp) of each N-tile range
  float* tgt;                       // [s]: target logit
  Header* hdr;
  // gradient epilogue only
  const float* lse;                 // [s] logsumexp of the forward
  const float* grad_rows;           // [s] per-row upstream gradient, or null
  float grad;                       // upstream gradient g of the reduced loss (grad_rows null)
  unsigned short* dz;               // [s, ldz] bf16 dlogits, shard i's column j at dz + dzcol[i] + j
  long long ldz;
  int dzcol[kMaxGemmShards + 1];
  // logits-keeping epilogue only: shard i's fp32 logits [s, w_i], box 32 x 32
  CUtensorMap tmz[kMaxGemmShards];
};

constexpr int kEpiStats = 0;  // loss statistics of the tile
constexpr int kEpiGrad = 1;   // dlogits of the tile, from the forward's logsumexp
constexpr int kEpiStatsZ = 2; // loss statistics of the tile, and the tile's fp32 logits kept

// The logits-keeping epilogue stages each warp's 32 rows x 32 columns of fp32
// (4 KB, 128-byte swizzle) in shared memory past GemmSmem, two buffers per
// warp, and stores them with TMA: a thread's row is 128 contiguous bytes, so
// plain stores from registers would touch 32 lines per warp instruction.
constexpr int kZStageOff = int((sizeof(GemmSmem) + 1023) / 1024 * 1024);
constexpr int kZWarpBytes = 2 * 4096;
constexpr int kZSmem = kZStageOff + 4 * kZWarpBytes;
static_assert(kZSmem <= 232448, "logits staging fits the shared memory of a CTA");

using namespace tc;

// Instruction descriptor of the logits product: M = kBM, N = kBN, X and W_i
// both K-major.
constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN, false, false);

__device__ __forceinline__ int shard_of_tile(const GemmParams& p, int nt) {
  int i = 0;
  while (p.nstart[i + 1] <= nt) ++i;
  return i;
}

// One epilogue row: the running statistics of the row's columns this CTA
// covers, and for the gradient epilogue the row's exponent offset and scale.
struct EpiRow {
  int r;
  bool live;
  long long y;
  float m, se, zt;
  bool has_t;
  float cb, scl;
};

template <int EPI>
__device__ __forceinline__ void epi_row_start(const GemmParams& p, int r, EpiRow& e) {
  e.r = r;
  e.live = r < p.s;
  e.y = e.live ? __ldg(p.targets + r) : -1;
  e.m = -INFINITY;
  e.se = 0.f;
  e.zt = 0.f;
  e.has_t = false;
  e.cb = 0.f;  // gradient epilogue: 0 for rows outside the batch or ignored
  e.scl = 0.f;
  if (EPI == kEpiGrad && e.live && e.y != p.ignore_index) {
    // the forward's header: g / n_valid for 'mean', g otherwise
    const int nv = p.hdr->n_valid;
    const float sc_all = p.hdr->reduction != VPCE_MEAN ? p.grad : (nv > 0 ? p.grad / float(nv) : 0.f);
    e.cb = -__ldg(p.lse + r) * kLog2e;
    e.scl = p.grad_rows != nullptr ? __ldg(p.grad_rows + r) : sc_all;
  }
}

// The 256 columns of one accumulator for one row (TMEM columns from
// `acc_addr`): statistics, plus the kept logits or the dlogits by EPI.
template <int EPI>
__device__ __forceinline__ void epi_row_tile(const GemmParams& p, EpiRow& e, uint32_t acc_addr, int sh, int col0,
                                             int valid, int mt, int q, int lane, unsigned& zc,
                                             unsigned char* zbuf) {
  const long long tc = e.y - (long long)p.vstart[sh] - col0;  // target column inside this tile
  if constexpr (EPI == kEpiGrad) {
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      if (c * 32 >= valid) break;  // warp-uniform
      float v[32];
      tmem_ld32(acc_addr + uint32_t(c * 32), v);
      const int lim = valid - c * 32;
      const long long rel = tc - c * 32;
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        // (softmax - onehot) * g, rounded to nearest-even bf16
        float d0 = ex2(fmaf(v[j], kLog2e, e.cb)) * e.scl;
        float d1 = ex2(fmaf(v[j + 1], kLog2e, e.cb)) * e.scl;
        if (j == rel) d0 -= e.scl;
        if (j + 1 == rel) d1 -= e.scl;
        if (e.scl == 0.f) d0 = d1 = 0.f;  // ignored or padding rows (also keeps inf * 0 out)
        w[j / 2] = pack_bf16x2(d0, d1);
      }
      if (e.live) {
        const long long col = (long long)p.dzcol[sh] + col0 + c * 32;
        unsigned short* dst = p.dz + (long long)e.r * p.ldz + col;
        if (lim == 32 && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < lim) dst[j] = (unsigned short)((j & 1) ? (w[j / 2] >> 16) : (w[j / 2] & 0xffffu));
        }
      }
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      if (c * 32 >= valid) break;  // warp-uniform
      float v[32];
      tmem_ld32(acc_addr + uint32_t(c * 32), v);
      const int lim = valid - c * 32;
      const long long rel = tc - c * 32;
      if constexpr (EPI == kEpiStatsZ) {
        // this warp's 32 rows x 32 columns through shared memory to the
        // shard's kept logits; TMA clips columns past the shard and rows
        // past the chunk.  A warp whose rows all lie past the chunk stages
        // nothing (warp-uniform), so that zc counts exactly the stores
        // issued and the buffer-reuse wait below covers the right one.
        const int zy = mt * kBM + q * 32;
        if (zy < p.s) {
          unsigned char* zb = zbuf + (zc & 1u) * 4096u;
          if (lane == 0 && zc >= 2) bulk_wait_read<1>();  // the store of chunk zc - 2 has read zb
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(zb + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmz[sh], zb, col0 + c * 32, zy);
            bulk_commit();
          }
          ++zc;
        }
      }
      if (rel >= 0 && rel < 32 && rel < lim) {
        // the target logit: a sum of products with 0/1 weights picks it
        // without a run-time index into the registers (exact: one term is
        // 1 * z, the rest are 0 * finite)
        float pick = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) pick = fmaf(j == int(rel) ? 1.f : 0.f, v[j], pick);
        e.zt = pick;
        e.has_t = true;
      }
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j >= lim) v[j] = -INFINITY;
        cm = fmaxf(cm, v[j]);
      }
      if (cm > e.m) {
        e.se *= ex2((e.m - cm) * kLog2e);
        e.m = cm;
      }
      const float nb = -e.m * kLog2e;
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        a0 += ex2(fmaf(v[j], kLog2e, nb));
        a1 += ex2(fmaf(v[j + 1], kLog2e, nb));
      }
      e.se += a0 + a1;
    }
  }
}

// The N tiles group grp takes in wave wv, and the index of that range (the
// partial it writes).  The gn ranges split the N tiles as evenly as integer
// division allows, and a group's range moves on by one each wave.  The ranges
// one tile longer than the rest then fall to each group in turn, so that no
// CTA runs more than the ceiling of the mean tile count over all waves.
__device__ __forceinline__ int wave_range(const GemmParams& p, int grp, int wv, int* nt0, int* nt1) {
  const int g = (grp + wv) % p.gn;
  *nt0 = int((long long)g * p.n_tiles / p.gn);
  *nt1 = int((long long)(g + 1) * p.n_tiles / p.gn);
  return g;
}

template <int EPI>
__device__ __forceinline__ void epi_row_finish(const GemmParams& p, const EpiRow& e, int range) {
  if (EPI != kEpiGrad && e.live) {
    p.part[(long long)range * p.s + e.r] = make_float2(e.m, e.se);
    if (e.has_t) p.tgt[e.r] = e.zt;
  }
}

template <int EPI>
__global__ void __launch_bounds__(kGThreads, 1) gemm_stats_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, 4);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  const int m_slot = int(blockIdx.x) % p.gm;
  const int grp = int(blockIdx.x) / p.gm;
  const int waves = (p.m_pairs + p.gm - 1) / p.gm;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      unsigned issued = 0;
      bool ok = true;
      for (int wv = 0; wv < waves && ok; ++wv) {
        const int mp = wv * p.gm + m_slot;
        if (mp >= p.m_pairs) break;
        int nt0, nt1;
        wave_range(p, grp, wv, &nt0, &nt1);
        for (int nt = nt0; nt < nt1 && ok; ++nt) {
          const int sh = shard_of_tile(p, nt);
          const int n_off = (nt - p.nstart[sh]) * kBN;
          for (int kb = 0; kb < p.k_steps; ++kb) {
            const int st = int(issued % kGStages);
            if (!wait1(&sm.empty[st], ((issued / kGStages) & 1u) ^ 1u, &sm.abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.full[st], kGStage);
            // the pair's X tiles (the second reads zeros past the last row
            // when the M tiles are odd) and the shared W tile
#pragma unroll
            for (int j = 0; j < kMT; ++j)
              tma_load_2d(sm.stage[st] + j * kATile, &p.tmx, kb * kBK, (kMT * mp + j) * kBM, &sm.full[st]);
            tma_load_2d(sm.stage[st] + kMT * kATile, &p.tmw[sh], kb * kBK, n_off, &sm.full[st]);
            ++issued;
          }
        }
      }
      if (!ok) {
        sm.abort_flag = 1;
        atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
        // the copies still in flight land in shared memory before the CTA exits
        const unsigned first = issued > unsigned(kGStages) ? issued - kGStages : 0u;
        for (unsigned j = first; j < issued; ++j) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&sm.full[j % kGStages], (j / kGStages) & 1u) && clock64() - t0 < kWaitLimitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      unsigned consumed = 0, tiles = 0, issued_any = 0;
      bool ok = true;
      for (int wv = 0; wv < waves && ok; ++wv) {
        const int mp = wv * p.gm + m_slot;
        if (mp >= p.m_pairs) break;
        int nt0, nt1;
        wave_range(p, grp, wv, &nt0, &nt1);
        for (int nt = nt0; nt < nt1 && ok; ++nt) {
          // the epilogue has read the previous tile's accumulators
          if (!wait1(&sm.acc_empty, (tiles & 1u) ^ 1u, &sm.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < p.k_steps; ++kb) {
            const int st = int(consumed % kGStages);
            if (!wait1(&sm.full[st], (consumed / kGStages) & 1u, &sm.abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_addr(sm.stage[st]);
            const uint32_t b0 = a0 + kMT * kATile;
#pragma unroll
            for (int kk = 0; kk < kBK / kUK; ++kk) {
              const uint64_t bdesc = sw128_desc(b0 + kk * kUK * 2);
#pragma unroll
              for (int j = 0; j < kMT; ++j)
                umma_bf16(tmem + uint32_t(j * kBN), sw128_desc(a0 + j * kATile + kk * kUK * 2), bdesc, kIdesc,
                          (kb | kk) != 0);
            }
            issued_any = 1;
            umma_commit(&sm.empty[st]);  // the stage is free once these MMAs have read it
            ++consumed;
          }
          if (!ok) break;
          umma_commit(&sm.acc_full);  // the pair's accumulators are complete
          ++tiles;
        }
      }
      if (!ok) {
        sm.abort_flag = 1;
        atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
      }
      if (issued_any) {  // every MMA has finished before the TMEM is released
        umma_commit(&sm.drain);
        const long long t0 = clock64();
        while (!mbar_try_wait(&sm.drain, 0u) && clock64() - t0 < kWaitLimitCycles) {
        }
      }
    }
  } else {
    // ---------------- epilogue: one row of each M tile per thread
    const int q = warp & 3;  // the TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    const uint32_t lane_addr = tmem + (uint32_t(q * 32) << 16);
    unsigned tiles = 0;
    bool ok = true;
    unsigned zc = 0;  // chunks this warp has staged (logits-keeping epilogue)
    unsigned char* zbuf = smem_raw + kZStageOff + q * kZWarpBytes;
    for (int wv = 0; wv < waves && ok; ++wv) {
      const int mp = wv * p.gm + m_slot;
      if (mp >= p.m_pairs) break;
      int nt0, nt1;
      const int range = wave_range(p, grp, wv, &nt0, &nt1);
      EpiRow e0, e1;
      epi_row_start<EPI>(p, (kMT * mp) * kBM + row_in_tile, e0);
      epi_row_start<EPI>(p, (kMT * mp + 1) * kBM + row_in_tile, e1);
      for (int nt = nt0; nt < nt1; ++nt) {
        if (!waitw(&sm.acc_full, tiles & 1u, &sm.abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int sh = shard_of_tile(p, nt);
        const int col0 = (nt - p.nstart[sh]) * kBN;
        const int width = p.vstart[sh + 1] - p.vstart[sh];
        const int valid = min(kBN, width - col0);
        epi_row_tile<EPI>(p, e0, lane_addr, sh, col0, valid, kMT * mp, q, lane, zc, zbuf);
        epi_row_tile<EPI>(p, e1, lane_addr + uint32_t(kBN), sh, col0, valid, kMT * mp + 1, q, lane, zc, zbuf);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_local(&sm.acc_empty);
        ++tiles;
      }
      if (!ok) break;
      epi_row_finish<EPI>(p, e0, range);
      epi_row_finish<EPI>(p, e1, range);
    }
    if (!ok && lane == 0) {
      sm.abort_flag = 1;
      atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
    }
    if (EPI == kEpiStatsZ && lane == 0) bulk_wait_all<0>();  // the staged logits have left shared memory
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    tmem_dealloc(tmem, kTmemCols);
}

// A [rows, h] bf16 row-major matrix (row stride ld elements) as a 2-D tensor
// map with a box of 64 columns x box_rows rows and the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, long long h, long long ld, int box_rows) {
  return make_map_bf16(m, base, rows, h, ld, kBK, box_rows);
}

}  // namespace

int gemm_max_shards() { return kMaxGemmShards; }
int gemm_max_groups(int sms) { return sms > 0 ? sms : 1; }

cudaError_t set_gemm_smem() {
  const cudaError_t e = cudaFuncSetAttribute(gemm_stats_kernel<kEpiStats>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(GemmSmem)));
  if (e != cudaSuccess) return e;
  const cudaError_t e2 = cudaFuncSetAttribute(gemm_stats_kernel<kEpiStatsZ>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, kZSmem);
  if (e2 != cudaSuccess) return e2;
  return cudaFuncSetAttribute(gemm_stats_kernel<kEpiGrad>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(sizeof(GemmSmem)));
}

// The grid of the fused LM-head kernel for s rows and n_tiles N tiles on sms
// SMs: gm M tiles per wave share each W tile, gn groups split the N tiles.
// gm M-tile pairs per wave (at most kMaxGroupsPerWave M tiles) times gn N
// groups: one CTA each, no more than the SMs.
void gemm_grid(long long s, int n_tiles, int sms, int* gm, int* gn) {
  const int m_pairs = int((s + kMT * kBM - 1) / (kMT * kBM));
  int a = m_pairs < kMaxGroupsPerWave / kMT ? m_pairs : kMaxGroupsPerWave / kMT;
  if (a < 1) a = 1;
  int b = sms / a;
  if (b > n_tiles) b = n_tiles;
  if (b < 1) b = 1;
  *gm = a;
  *gn = b;
}

int gemm_n_tiles(const long long* vocab_start, int t) {
  int n = 0;
  for (int i = 0; i < t; ++i) n += int((vocab_start[i + 1] - vocab_start[i] + kBN - 1) / kBN);
  return n;
}

// Encodes the tensor maps and launches the kernel; returns false when a
// tensor map cannot be encoded (the launch status is the caller's to read).
bool launch_gemm_stats(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                       long long h, const long long* vocab_start, const long long* targets, long long ignore_index,
                       float2* part, float* tgt, Header* hdr, int sms, int* groups, cudaStream_t st, float* zf,
                       long long ldzf, const long long* zcol) {
  static_assert(sizeof(GemmParams) < 32000, "kernel parameter block");
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_map(&p.tmx, x, s, h, ld_x, kBM)) return false;
  p.nstart[0] = 0;
  for (int i = 0; i < t; ++i) {
    const long long wi = vocab_start[i + 1] - vocab_start[i];
    if (!make_map(&p.tmw[i], w[i], wi, h, ld_w, kBN)) return false;
    p.vstart[i] = int(vocab_start[i]);
    p.nstart[i + 1] = p.nstart[i] + int((wi + kBN - 1) / kBN);
  }
  p.vstart[t] = int(vocab_start[t]);
  p.t = t;
  p.s = int(s);
  p.k_steps = int(h / kBK);
  p.m_tiles = int((s + kBM - 1) / kBM);
  p.m_pairs = (p.m_tiles + kMT - 1) / kMT;
  p.n_tiles = p.nstart[t];
  gemm_grid(s, p.n_tiles, sms, &p.gm, &p.gn);
  p.targets = targets;
  p.ignore_index = ignore_index;
  p.part = part;
  p.tgt = tgt;
  p.hdr = hdr;
  *groups = p.gn;
  if (zf != nullptr) {
    // shard i's logits at columns [zcol[i], zcol[i] + w_i) of rows of ldzf
    // floats (zcol[i] a multiple of 4, ldzf a multiple of 4)
    for (int i = 0; i < t; ++i)
      if (!make_map_f32(&p.tmz[i], zf + zcol[i], s, vocab_start[i + 1] - vocab_start[i], ldzf)) return false;
    gemm_stats_kernel<kEpiStatsZ><<<p.gm * p.gn, kGThreads, kZSmem, st>>>(p);
  }
  else
    gemm_stats_kernel<kEpiStats><<<p.gm * p.gn, kGThreads, sizeof(GemmSmem), st>>>(p);
  return true;
}

// dlogits of rows [0, s) of X (the caller offsets X, targets, lse and
// grad_rows to a chunk), written as bf16 into dz (row stride ldz elements;
// shard i's column j of a row at dz + zcol[i] + j).
bool launch_gemm_grad(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                      long long h, const long long* vocab_start, const long long* targets, long long ignore_index,
                      const float* lse, const float* grad_rows, float grad, unsigned short* dz, long long ldz,
                      const long long* zcol, Header* hdr, int sms, cudaStream_t st) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_map(&p.tmx, x, s, h, ld_x, kBM)) return false;
  for (int i = 0; i < t; ++i) {
    const long long wi = vocab_start[i + 1] - vocab_start[i];
    if (!make_map(&p.tmw[i], w[i], wi, h, ld_w, kBN)) return false;
    p.vstart[i] = int(vocab_start[i]);
    p.nstart[i + 1] = p.nstart[i] + int((wi + kBN - 1) / kBN);
  }
  p.vstart[t] = int(vocab_start[t]);
  p.t = t;
  p.s = int(s);
  p.k_steps = int(h / kBK);
  p.m_tiles = int((s + kBM - 1) / kBM);
  p.m_pairs = (p.m_tiles + kMT - 1) / kMT;
  p.n_tiles = p.nstart[t];
  gemm_grid(s, p.n_tiles, sms, &p.gm, &p.gn);
  p.targets = targets;
  p.ignore_index = ignore_index;
  p.hdr = hdr;
  p.lse = lse;
  p.grad_rows = grad_rows;
  p.grad = grad;
  p.dz = dz;
  p.ldz = ldz;
  for (int i = 0; i <= t; ++i) p.dzcol[i] = int(zcol[i]);
  gemm_stats_kernel<kEpiGrad><<<p.gm * p.gn, kGThreads, sizeof(GemmSmem), st>>>(p);
  return true;
}

}  // namespace vpce
