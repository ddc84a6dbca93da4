// The two products of the LM-head backward on the tensor cores, for one
// chunk of R rows whose dZ = dL/dz (bf16, rows of ldz elements, shard i's
// columns from column zcol[i]) is already formed:
//     dX      = sum_i dZ_i W_i        [R, h]    bf16, written
//     dW_i   += dZ_i^T X              [w_i, h]  fp32, accumulated
// The pages give no backward; this is the chain rule through z_i = X W_i^T
// (the head split by vocabulary as in "LLM Internals" §7.3.4), with the
// vocabulary-sharded contraction of dX running over every shard inside one
// accumulator, so no per-shard partial of dX is ever stored.
//
// Kernel shape: the logits kernel's (one persistent 192-thread CTA per SM, a
// pair of 128-row M tiles against one 256-column N tile, 3 stages of 64 KB,
// 512 TMEM columns for the pair's fp32 accumulators), with operands in the
// layouts the data already has:
//   dX   A = dZ rows, K (vocabulary) contiguous: K-major, as the logits' X;
//        B = W_i [w_i, h]: each K row (vocabulary entry) holds N (h)
//        contiguous: MN-major, four 64-column blocks per 256-wide tile.  The
//        K loop runs over every shard's 64-deep steps in order.
//   dW   A = dZ_i^T: a K row (token) holds M (vocabulary) contiguous:
//        MN-major; B = X [R, h]: MN-major.  K runs over the chunk's rows.
//   warp 0      TMA loads (128-byte swizzle; MN-major operands as 64 x 64
//               boxes, one 8 KB block per 64 columns of M or N);
//   warp 1      TMEM allocation and the MMA issue (M = 128, N = 256, K = 16
//               per tcgen05.mma, two per K slice sharing the B tile);
//   warps 2..5  the epilogue, one TMEM lane (an output row) per thread: dX
//               rounds to bf16 and stores its row's 256 columns; dW stages
//               32 x 32 fp32 blocks per warp in swizzled shared memory and
//               adds them into dW_i with TMA tile reductions (the adds happen
//               at L2, each dW element gets exactly one add per chunk, so the
//               result is the same on every run).
// Ragged edges come from the TMA's zero fill (K past a shard's width or the
// chunk's rows, M past the rows or the shard, N past h); stores and
// reductions are clipped to the tensors' extents.
#include <cstring>

#include "vpce_kernels.cuh"
#include "vpce_tc.cuh"

namespace vpce {

namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kUK = 16;
constexpr int kMT = 2;  // M tiles per CTA tile, sharing each B tile
constexpr int kStages = 3;
constexpr int kATile = kBM * kBK * 2;    // 16 KB
constexpr int kBTile = kBN * kBK * 2;    // 32 KB
constexpr int kStage = kMT * kATile + kBTile;
constexpr int kMnBlock = 64 * kBK * 2;   // 8 KB: 64 columns of M or N by 64 K rows (MN-major)
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kMaxShards = 32;

constexpr int kDX = 0;
constexpr int kDW = 1;

struct BwdSmem {
  unsigned char stage[kStages][kStage];  // 1024-byte aligned: A0, A1, B
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// dW epilogue: two 32 x 32 fp32 staging blocks (4 KB each, 128-byte swizzle)
// per epilogue warp past BwdSmem.
constexpr int kRedOff = int((sizeof(BwdSmem) + 1023) / 1024 * 1024);
constexpr int kRedWarpBytes = 2 * 4096;
constexpr int kSmemDW = kRedOff + 4 * kRedWarpBytes;
static_assert(kSmemDW <= 232448, "dW staging fits the shared memory of a CTA");

struct BwdParams {
  CUtensorMap tma[kMaxShards];  // dZ of shard i [R, w_i]: dX box 64 x 128 (K-major), dW box 64 x 64 (M-major)
  CUtensorMap tmb[kMaxShards];  // dX: W_i [w_i, h], box 64 x 64; dW: tmb[0] = X [R, h], box 64 x 64
  CUtensorMap tmd[kMaxShards];  // dW: dW_i [w_i, h] fp32, box 32 x 32
  int t;
  int R;
  int h;
  int n_tiles;                  // ceil(h / kBN)
  int m_pairs;                  // dX: ceil(R / (kMT kBM))
  int k_steps;                  // dX: sum of ceil(w_i / kBK); dW: ceil(R / kBK)
  int kstart[kMaxShards + 1];   // dX: first K step of shard i
  int pstart[kMaxShards + 1];   // dW: first M-tile pair of shard i (pairs of 256 vocabulary rows)
  int width[kMaxShards];        // w_i
  int tiles;
  int group;                    // M-tile pairs per raster group
  unsigned short* dx;           // dX: bf16 [R, ld_dx]
  long long ld_dx;
  Header* hdr;
};

constexpr uint32_t kIdescDX = idesc_bf16(kBM, kBN, false, true);
constexpr uint32_t kIdescDW = idesc_bf16(kBM, kBN, true, true);

// Tile k of the walk.  The M-tile pairs (counted over all shards for dW) run
// in groups of p.group: within a group the N tiles in order, the group's
// pairs fastest.  The CTAs that run at the same time then share both their A
// blocks (the group's pairs) and their B blocks (a few N tiles), so each
// block comes from HBM about once per group instead of once per wave.
struct Tile {
  int sh, mp, nt;
};

template <int MODE>
__device__ __forceinline__ Tile tile_at(const BwdParams& p, int k) {
  const int total = MODE == kDX ? p.m_pairs : p.pstart[p.t];
  const int per_group = p.group * p.n_tiles;
  const int g = k / per_group;
  const int j = k - g * per_group;
  const int first = g * p.group;
  const int gsize = min(p.group, total - first);
  Tile tl;
  tl.nt = j / gsize;
  const int q = first + (j - tl.nt * gsize);
  if (MODE == kDX) {
    tl.sh = 0;
    tl.mp = q;
  } else {
    int i = 0;
    while (p.pstart[i + 1] <= q) ++i;
    tl.sh = i;
    tl.mp = q - p.pstart[i];
  }
  return tl;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) gemm_bwd_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, 4);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      unsigned issued = 0;
      bool ok = true;
      for (int k = blockIdx.x; k < p.tiles && ok; k += gridDim.x) {
        const Tile tl = tile_at<MODE>(p, k);
        int sh = 0;
        for (int ks = 0; ks < p.k_steps; ++ks) {
          const int st = int(issued % kStages);
          if (!wait1(&sm.empty[st], ((issued / kStages) & 1u) ^ 1u, &sm.abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.full[st], kStage);
          unsigned char* a = sm.stage[st];
          unsigned char* b = a + kMT * kATile;
          if (MODE == kDX) {
            while (p.kstart[sh + 1] <= ks) ++sh;
            const int kx = (ks - p.kstart[sh]) * kBK;  // vocabulary column inside shard sh
#pragma unroll
            for (int j = 0; j < kMT; ++j)
              tma_load_2d(a + j * kATile, &p.tma[sh], kx, (kMT * tl.mp + j) * kBM, &sm.full[st]);
#pragma unroll
            for (int c = 0; c < kBN / 64; ++c)
              tma_load_2d(b + c * kMnBlock, &p.tmb[sh], tl.nt * kBN + c * 64, kx, &sm.full[st]);
          } else {
            const int ky = ks * kBK;  // row of the chunk
#pragma unroll
            for (int j = 0; j < kMT; ++j)
#pragma unroll
              for (int c = 0; c < kBM / 64; ++c)
                tma_load_2d(a + j * kATile + c * kMnBlock, &p.tma[tl.sh], (kMT * tl.mp + j) * kBM + c * 64, ky,
                            &sm.full[st]);
#pragma unroll
            for (int c = 0; c < kBN / 64; ++c)
              tma_load_2d(b + c * kMnBlock, &p.tmb[0], tl.nt * kBN + c * 64, ky, &sm.full[st]);
          }
          ++issued;
        }
      }
      if (!ok) {
        sm.abort_flag = 1;
        atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
        // the copies still in flight land in shared memory before the CTA exits
        const unsigned first = issued > unsigned(kStages) ? issued - kStages : 0u;
        for (unsigned j = first; j < issued; ++j) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&sm.full[j % kStages], (j / kStages) & 1u) && clock64() - t0 < kWaitLimitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      unsigned consumed = 0, tiles = 0, issued_any = 0;
      bool ok = true;
      for (int k = blockIdx.x; k < p.tiles && ok; k += gridDim.x) {
        // the epilogue has read the previous tile's accumulators
        if (!wait1(&sm.acc_empty, (tiles & 1u) ^ 1u, &sm.abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < p.k_steps; ++ks) {
          const int st = int(consumed % kStages);
          if (!wait1(&sm.full[st], (consumed / kStages) & 1u, &sm.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(sm.stage[st]);
          const uint32_t b0 = a0 + kMT * kATile;
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk) {
            const uint64_t bdesc = sw128_mn_desc(b0 + kk * 2 * 1024, kMnBlock);
#pragma unroll
            for (int j = 0; j < kMT; ++j) {
              const uint64_t adesc = MODE == kDX ? sw128_desc(a0 + j * kATile + kk * kUK * 2)
                                                 : sw128_mn_desc(a0 + j * kATile + kk * 2 * 1024, kMnBlock);
              umma_bf16(tmem + uint32_t(j * kBN), adesc, bdesc, MODE == kDX ? kIdescDX : kIdescDW,
                        (ks | kk) != 0);
            }
          }
          issued_any = 1;
          umma_commit(&sm.empty[st]);  // the stage is free once these MMAs have read it
          ++consumed;
        }
        if (!ok) break;
        umma_commit(&sm.acc_full);  // the pair's accumulators are complete
        ++tiles;
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
    // ---------------- epilogue: one output row of each M tile per thread
    const int q = warp & 3;  // the TMEM lane quarter this warp may access
    const uint32_t lane_addr = tmem + (uint32_t(q * 32) << 16);
    unsigned tiles = 0;
    bool ok = true;
    unsigned zc = 0;  // staging blocks this warp has filled (dW)
    unsigned char* zbuf = smem_raw + kRedOff + q * kRedWarpBytes;
    for (int k = blockIdx.x; k < p.tiles; k += gridDim.x) {
      const Tile tl = tile_at<MODE>(p, k);
      if (!waitw(&sm.acc_full, tiles & 1u, &sm.abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int j = 0; j < kMT; ++j) {
        const int row0 = (kMT * tl.mp + j) * kBM + q * 32;  // this warp's first output row
        // rows past the chunk (dX) or the shard (dW) hold nothing to write;
        // skipping them here (warp-uniform) also keeps the staging buffers'
        // bulk-group count equal to the reductions issued
        if (row0 >= (MODE == kDX ? p.R : p.width[tl.sh])) continue;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          const int col = tl.nt * kBN + c * 32;
          if (col >= p.h) break;  // warp-uniform
          float v[32];
          tmem_ld32(lane_addr + uint32_t(j * kBN + c * 32), v);
          if (MODE == kDX) {
            const int r = row0 + lane;
            if (r < p.R) {
              uint32_t w[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
              unsigned short* dst = p.dx + (long long)r * p.ld_dx + col;
              if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                for (int u = 0; u < 4; ++u) d4[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) dst[e] = (unsigned short)((e & 1) ? (w[e / 2] >> 16) : (w[e / 2] & 0xffffu));
              }
            }
          } else {
            // this warp's 32 rows x 32 columns through shared memory, added
            // into dW_i by the TMA (rows past the shard are clipped)
            unsigned char* zb = zbuf + (zc & 1u) * 4096u;
            if (lane == 0 && zc >= 2) bulk_wait_read<1>();  // the reduction of block zc - 2 has read zb
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 8; ++e)
              *reinterpret_cast<float4*>(zb + lane * 128 + ((e ^ (lane & 7)) << 4)) =
                  make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&p.tmd[tl.sh], zb, col, row0);
              bulk_commit();
            }
            ++zc;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_local(&sm.acc_empty);
      ++tiles;
    }
    if (!ok && lane == 0) {
      sm.abort_flag = 1;
      atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
    }
    if (MODE == kDW && lane == 0) bulk_wait_all<0>();  // every reduction has completed
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t set_gemm_bwd_smem() {
  const cudaError_t e =
      cudaFuncSetAttribute(gemm_bwd_kernel<kDX>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(BwdSmem)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_bwd_kernel<kDW>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemDW);
}

int gemm_bwd_max_shards() { return kMaxShards; }

// dX of one chunk: dx[r, :] (bf16, row stride ld_dx) = sum_i dZ_i[r, :] W_i for
// rows r < R.  dz + zcol[i] is shard i's first column (zcol[i] and ldz
// multiples of 8); W_i is [w_i, h] with row stride ld_w (a multiple of 8).
// Returns false when a tensor map cannot be encoded.
bool launch_dgrad_x(const unsigned short* dz, long long ldz, const long long* zcol, const void* const* w,
                    long long ld_w, int t, long long R, long long h, const long long* vs, void* dx, long long ld_dx,
                    Header* hdr, int sms, cudaStream_t st) {
  static_assert(sizeof(BwdParams) < 32000, "kernel parameter block");
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.kstart[0] = 0;
  for (int i = 0; i < t; ++i) {
    const long long wi = vs[i + 1] - vs[i];
    if (!make_map_bf16(&p.tma[i], dz + zcol[i], R, wi, ldz, kBK, kBM)) return false;
    if (!make_map_bf16(&p.tmb[i], w[i], wi, h, ld_w, 64, kBK)) return false;
    p.width[i] = int(wi);
    p.kstart[i + 1] = p.kstart[i] + int((wi + kBK - 1) / kBK);
  }
  p.t = t;
  p.R = int(R);
  p.h = int(h);
  p.n_tiles = int((h + kBN - 1) / kBN);
  p.m_pairs = int((R + kMT * kBM - 1) / (kMT * kBM));
  p.k_steps = p.kstart[t];
  p.tiles = p.m_pairs * p.n_tiles;
  // groups of 8 pairs: 18.3 GB of reads per full-size launch against 17.2 for one pair per
  // group, but the sustained training step is 1.5 % faster (31.0 against 31.5 ms, six
  // interleaved runs of ten steps)
  p.group = 8;
  p.dx = static_cast<unsigned short*>(dx);
  p.ld_dx = ld_dx;
  p.hdr = hdr;
  const int grid = p.tiles < sms ? p.tiles : sms;
  gemm_bwd_kernel<kDX><<<grid, kThreads, sizeof(BwdSmem), st>>>(p);
  return true;
}

// dW of one chunk: dw[i][v, :] (fp32, row stride ld_dw, a multiple of 4) +=
// sum over the chunk's rows r of dZ_i[r, v] X[r, :]; X is [R, h] with row
// stride ld_x (a multiple of 8).
bool launch_dgrad_w(const unsigned short* dz, long long ldz, const long long* zcol, const void* x, long long ld_x,
                    int t, long long R, long long h, const long long* vs, float* const* dw, long long ld_dw,
                    Header* hdr, int sms, cudaStream_t st) {
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_map_bf16(&p.tmb[0], x, R, h, ld_x, 64, kBK)) return false;
  p.pstart[0] = 0;
  for (int i = 0; i < t; ++i) {
    const long long wi = vs[i + 1] - vs[i];
    if (!make_map_bf16(&p.tma[i], dz + zcol[i], R, wi, ldz, 64, kBK)) return false;
    if (!make_map_f32(&p.tmd[i], dw[i], wi, h, ld_dw)) return false;
    p.width[i] = int(wi);
    p.pstart[i + 1] = p.pstart[i] + int((wi + kMT * kBM - 1) / (kMT * kBM));
  }
  p.t = t;
  p.R = int(R);
  p.h = int(h);
  p.n_tiles = int((h + kBN - 1) / kBN);
  p.k_steps = int((R + kBK - 1) / kBK);
  p.tiles = p.pstart[t] * p.n_tiles;
  p.group = 16;  // measured: 17.7 GB of reads per full-size launch against 19.7 (8) and 22.4 (32)
  p.hdr = hdr;
  const int grid = p.tiles < sms ? p.tiles : sms;
  gemm_bwd_kernel<kDW><<<grid, kThreads, kSmemDW, st>>>(p);
  return true;
}

}  // namespace vpce
