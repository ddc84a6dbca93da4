// Fused forward + backward of the vocab-parallel cross-entropy: the loss and
// the in-place dlogits in one pass over HBM.
//
// The method ("Distributed Training III: Model Parallelism", CMU 11-868
// Lecture 16 notes, §5.5; "LLM Internals" §7.3.4) reduces per row the maximum,
// the sum of exponentials and the target logit over the vocabulary shards and
// combines them into logsumexp - target.  When the upstream gradient g is known
// up front (the loss is the last op, g = 1 or a loss scale), the backward of a
// row can follow its forward immediately, while the row is still on chip:
//
//   * a group of G warps owns one row at a time; each warp takes a 1/G
//     sub-range of every shard segment of that row;
//   * pass 1 streams the sub-ranges from HBM through the warp's shared-memory
//     ring (cp.async.bulk + mbarrier) and keeps an online (max, sum-exp);
//   * the G warps meet at a per-row mbarrier, merge their partials in warp
//     order (every warp gets the same logsumexp) -- the on-chip stand-in for
//     the pages' max / sum / target all-reduces;
//   * pass 2 streams the same bytes again -- now L2 hits, the row was read
//     microseconds earlier -- turns them into dlogits in shared memory and
//     writes them back over the logits with cp.async.bulk stores.
//
// HBM sees one read and one write of the logits instead of two reads and one
// write.  The batch count n_valid (needed for the 1/n_valid of the mean before
// any gradient is written) comes from a one-block prologue kernel that also
// clears the workspace header; the batch loss is summed in a fixed order by the
// last block to finish.
#include "vpce_chunk.cuh"

namespace vpce {

namespace {

constexpr int kFusedWarps = 8;
constexpr int kPrepThreads = 1024;
constexpr int kFChunk = 4096;  // bytes per pipeline chunk
constexpr int kRingA = 4;      // pass-1 (HBM) slots per warp
constexpr int kRingB = 3;      // pass-2 (L2) slots per warp

struct FusedParams {
  ShardSet sh;
  int t;
  long long s;
  long long V;
  const long long* targets;
  long long ignore_index;
  int reduction;
  float grad;
  float* lse;        // [s]
  float* rowl;       // [s]: per-row loss (0 ignored, NaN bad target)
  float* row_loss;   // optional user copy of rowl
  float* loss_out;
  Header* hdr;
};

// Prologue: clear the header, count the valid rows, flag bad targets.
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const long long* targets, long long s,
                                                            long long V, long long ignore_index, Header* hdr,
                                                            int reduction, float* loss_out) {
  __shared__ int sc[kPrepThreads / 32];
  __shared__ int sbad[kPrepThreads / 32];
  int c = 0, bad = 0;
  for (long long r = threadIdx.x; r < s; r += kPrepThreads) {
    const long long y = targets[r];
    if (y == ignore_index) continue;
    if (y < 0 || y >= V) bad = 1;
    else ++c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    c += __shfl_down_sync(kFull, c, o);
    bad |= __shfl_down_sync(kFull, bad, o);
  }
  if ((threadIdx.x & 31) == 0) {
    sc[threadIdx.x >> 5] = c;
    sbad[threadIdx.x >> 5] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tc = 0, tb = 0;
    for (int i = 0; i < kPrepThreads / 32; ++i) {
      tc += sc[i];
      tb |= sbad[i];
    }
    hdr->n_valid = tc;
    hdr->error_flag = tb ? VPCE_FLAG_BAD_TARGET : 0;
    hdr->ticket = 0u;
    hdr->reduction = reduction;
    hdr->loss_sum = 0.0;
    if (s == 0) *loss_out = reduction == VPCE_SUM ? 0.f : __int_as_float(0x7fc00000);
  }
}

// Byte range [lo, hi) of shard segment `i` owned by warp `wg` of a group of G
// (16-byte boundaries; the last warp takes the remainder).
template <int G>
__device__ __forceinline__ void sub_range(unsigned seg_bytes, int wg, unsigned& lo, unsigned& hi) {
  lo = unsigned((unsigned long long)seg_bytes * unsigned(wg) / G) & ~15u;
  hi = wg == G - 1 ? seg_bytes : unsigned((unsigned long long)seg_bytes * unsigned(wg + 1) / G) & ~15u;
}

// Walks the chunks of one row that belong to warp wg: segment by segment,
// each sub-range cut into near-equal 16-byte aligned chunks of at most kFChunk.
template <int G, int EB>
struct RowWalk {
  int seg;
  unsigned k, n, lo, hi;
  bool ok;

  __device__ __forceinline__ bool seek(const FusedParams& p, int wg, int from) {
    for (seg = from; seg < p.t; ++seg) {
      sub_range<G>(unsigned(p.sh.start[seg + 1] - p.sh.start[seg]) * EB, wg, lo, hi);
      n = (hi - lo + kFChunk - 1) / kFChunk;
      if (n > 0) {
        k = 0;
        return ok = true;
      }
    }
    return ok = false;
  }
  __device__ __forceinline__ void next(const FusedParams& p, int wg) {
    if (++k < n) return;
    seek(p, wg, seg + 1);
  }
  // byte range [a, b) of the current chunk within its segment's row
  __device__ __forceinline__ void bounds(unsigned& a, unsigned& b) const {
    const unsigned len = hi - lo;
    a = lo + (unsigned((unsigned long long)len * k / n) & ~15u);
    b = k + 1 == n ? hi : lo + (unsigned((unsigned long long)len * (k + 1) / n) & ~15u);
  }
  __device__ __forceinline__ unsigned char* addr(const FusedParams& p, long long r, unsigned a) const {
    return const_cast<unsigned char*>(p.sh.ptr[seg]) + r * p.sh.ld_bytes[seg] + a;
  }
};

// Pass-1 chunk sequence of one warp across the rows of its group (ignored
// rows and rows without chunks for this warp are skipped).
template <int G, int EB>
struct RowsWalk {
  long long r, r_step;
  RowWalk<G, EB> w;
  bool ok;

  __device__ __forceinline__ void seek_row(const FusedParams& p, int wg, long long from) {
    ok = false;
    for (r = from; r < p.s; r += r_step) {
      if (__ldg(p.targets + r) == p.ignore_index) continue;
      if (w.seek(p, wg, 0)) {
        ok = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void next(const FusedParams& p, int wg) {
    w.next(p, wg);
    if (!w.ok) seek_row(p, wg, r + r_step);
  }
};

template <typename T, int G>
__global__ void __launch_bounds__(kFusedWarps * 32, 1) fused_kernel(const __grid_constant__ FusedParams p) {
  constexpr int EB = Elem<T>::kBytes;
  constexpr int NG = kFusedWarps / G;   // row groups per block
  constexpr int VPL = kFChunk / 512;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = warp / G, wg = warp % G;

  // shared memory: pass-1 rings [warps][kRingA] | pass-2 rings [warps][kRingB]
  // | slot barriers | row barriers [NG][2] | row partials [NG][2][G]
  unsigned char* ringA = smem + size_t(warp) * kRingA * kFChunk;
  unsigned char* ringB = smem + size_t(kFusedWarps) * kRingA * kFChunk + size_t(warp) * kRingB * kFChunk;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(kFusedWarps) * (kRingA + kRingB) * kFChunk);
  uint64_t* barA = bars + warp * (kRingA + kRingB);
  uint64_t* barB = barA + kRingA;
  uint64_t* rowbar = bars + kFusedWarps * (kRingA + kRingB) + grp * 2;
  float2* red = reinterpret_cast<float2*>(bars + kFusedWarps * (kRingA + kRingB) + NG * 2) + grp * 2 * G;
  __shared__ bool last;
  __shared__ double sv[kFusedWarps];

  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kRingA + kRingB; ++k) mbar_init(&barA[k], 1);
    if (wg == 0) {
      mbar_init(&rowbar[0], G);
      mbar_init(&rowbar[1], G);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int n_valid = p.hdr->n_valid;
  const float scale = p.reduction == VPCE_SUM ? p.grad : (n_valid > 0 ? p.grad / float(n_valid) : 0.f);
  const long long r_step = (long long)gridDim.x * NG;
  const long long r0 = (long long)blockIdx.x * NG + grp;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();

  // ring A streams pass-1 chunks from HBM kRingA ahead, across rows; the
  // lines are kept in L2 (evict_last) for pass 2
  RowsWalk<G, EB> prod;
  prod.r_step = r_step;
  prod.seek_row(p, wg, r0);
  unsigned issuedA = 0, kA = 0;
  auto issueA = [&](int slot) {
    unsigned a, b;
    prod.w.bounds(a, b);
    if (lane == 0) {
      mbar_arrive_expect_tx(&barA[slot], b - a);
      bulk_load(ringA + slot * kFChunk, prod.w.addr(p, prod.r, a), b - a, &barA[slot], pol_last);
    }
    ++issuedA;
    prod.next(p, wg);
  };
#pragma unroll 1
  for (int k = 0; k < kRingA && prod.ok; ++k) issueA(k);

  unsigned issuedB = 0, kB = 0, rounds = 0;
  bool alive = true;
#pragma unroll 1
  for (long long r = r0; r < p.s && alive; r += r_step) {
    const long long y = __ldg(p.targets + r);
    if (y == p.ignore_index) {
      // ignored row: zeros over this warp's sub-ranges, nothing read
      for (int i = 0; i < p.t; ++i) {
        unsigned lo, hi;
        sub_range<G>(unsigned(p.sh.start[i + 1] - p.sh.start[i]) * EB, wg, lo, hi);
        uint4* d = reinterpret_cast<uint4*>(const_cast<unsigned char*>(p.sh.ptr[i]) + r * p.sh.ld_bytes[i] + lo);
        for (unsigned v = lane; v < (hi - lo) >> 4; v += 32) d[v] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (wg == 0 && lane == 0) {
        p.rowl[r] = 0.f;
        p.lse[r] = 0.f;
        if (p.row_loss) p.row_loss[r] = 0.f;
      }
      continue;
    }
    const bool in_range = y >= 0 && y < p.V;
    // the target logit, read before any warp of the group can overwrite it
    float zt = 0.f;
    if (wg == 0 && lane == 0 && in_range) {
      int i = 0;
      while (p.sh.start[i + 1] <= y) ++i;
      zt = Elem<T>::load(p.sh.ptr[i] + r * p.sh.ld_bytes[i] + (y - p.sh.start[i]) * EB);
    }
    const int buf = int(rounds & 1u);
    const uint32_t rpar = (rounds >> 1) & 1u;
    ++rounds;

    // ---- pass 1: online (max, sum-exp) over this warp's sub-ranges
    float m = -INFINITY, sm = 0.f;
    RowWalk<G, EB> cw;
#pragma unroll 1
    for (cw.seek(p, wg, 0); cw.ok; cw.next(p, wg)) {
      unsigned a, b;
      cw.bounds(a, b);
      const int slot = int(kA % kRingA);
      if (!mbar_wait_warp(&barA[slot], (kA / kRingA) & 1u)) {
        alive = false;
        break;
      }
      stats_chunk<VPL>(ringA + slot * kFChunk, b - a, lane, m, sm, T());
      __syncwarp();
      if (prod.ok) issueA(slot);
      ++kA;
    }
    if (!alive) break;

    // ---- pass-2 loads (L2 hits) start now, while the group meets
    RowWalk<G, EB> iw;
    iw.seek(p, wg, 0);
    if (lane == 0) bulk_wait_read<0>();
#pragma unroll 1
    for (int k = 0; k < kRingB - 1 && iw.ok; ++k, iw.next(p, wg)) {
      unsigned a, b;
      iw.bounds(a, b);
      const int slot = int(issuedB % kRingB);
      if (lane == 0) {
        mbar_arrive_expect_tx(&barB[slot], b - a);
        bulk_load(ringB + slot * kFChunk, iw.addr(p, r, a), b - a, &barB[slot], pol_first);
      }
      ++issuedB;
    }

    warp_merge_ms(m, sm);
    float2* rd = red + buf * G;
    if (lane == 0) {
      rd[wg] = make_float2(m, sm);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&rowbar[buf])) : "memory");
    }
    if (!mbar_wait_warp(&rowbar[buf], rpar)) {
      alive = false;
      break;
    }
    // every warp folds the G partials in the same order -> the same lse
    float M = rd[0].x, S = rd[0].y;
#pragma unroll 1
    for (int j = 1; j < G; ++j) merge_ms(M, S, rd[j].x, rd[j].y);
    const float lse = in_range ? M + logf(S) : __int_as_float(0x7fc00000);
    if (wg == 0 && lane == 0) {
      const float rl = in_range ? lse - zt : lse;
      p.lse[r] = lse;
      p.rowl[r] = rl;
      if (p.row_loss) p.row_loss[r] = rl;
    }
    const float c = -lse * kLog2e;

    // ---- pass 2: dlogits in shared memory, bulk-stored over the logits
#pragma unroll 1
    for (cw.seek(p, wg, 0); cw.ok; cw.next(p, wg)) {
      unsigned a, b;
      cw.bounds(a, b);
      const int slot = int(kB % kRingB);
      if (!mbar_wait_warp(&barB[slot], (kB / kRingB) & 1u)) {
        alive = false;
        break;
      }
      unsigned char* sbuf = ringB + slot * kFChunk;
      const long long col0 = p.sh.start[cw.seg];
      const long long tb = (in_range && y >= col0 && y < p.sh.start[cw.seg + 1]) ? (y - col0) * EB : -1;
      const bool has_t = tb >= (long long)a && tb < (long long)b;
      float dt = 0.f;
      if (has_t && lane == 0) {
        const float z = Elem<T>::load(sbuf + (tb - a));
        dt = (ex2(fmaf(z, kLog2e, c)) - 1.f) * scale;
      }
      __syncwarp();
      grad_chunk<T, VPL>(sbuf, b - a, lane, c, scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (has_t) {
          Elem<T>::store(sbuf + (tb - a), dt);
          fence_proxy_async_smem();
        }
        bulk_store(cw.addr(p, r, a), sbuf, b - a, pol_first);
        bulk_commit();
      }
      if (iw.ok) {
        unsigned ia, ib;
        iw.bounds(ia, ib);
        const int ps = int(issuedB % kRingB);  // the slot of the previous chunk
        if (lane == 0) {
          bulk_wait_read<1>();
          mbar_arrive_expect_tx(&barB[ps], ib - ia);
          bulk_load(ringB + ps * kFChunk, iw.addr(p, r, ia), ib - ia, &barB[ps], pol_first);
        }
        ++issuedB;
        iw.next(p, wg);
      }
      ++kB;
    }
  }

  if (!alive) {
    if (lane == 0) atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
    for (unsigned k = kA; k < issuedA; ++k) {
      if (!mbar_wait_warp(&barA[k % kRingA], (k / kRingA) & 1u)) break;
    }
    for (unsigned k = kB; k < issuedB; ++k) {
      if (!mbar_wait_warp(&barB[k % kRingB], (k / kRingB) & 1u)) break;
    }
  }
  if (lane == 0) bulk_wait_all<0>();

  // ---- batch loss: the last block sums the per-row losses in a fixed order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&p.hdr->ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  double v = 0.0;
  // fixed 256-row blocks, each summed in row order by one thread, then a
  // fixed tree over the threads
  const long long nb = (p.s + 255) / 256;
  for (long long b = threadIdx.x; b < nb; b += kFusedWarps * 32) {
    double bs = 0.0;
    const long long e = min(p.s, (b + 1) * 256);
    for (long long r = b * 256; r < e; ++r) bs += double(__ldcg(p.rowl + r));
    v += bs;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(kFull, v, o);
  if (lane == 0) sv[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int i = 0; i < kFusedWarps; ++i) tot += sv[i];
    const int c = p.hdr->n_valid;
    p.hdr->loss_sum = tot;
    p.hdr->ticket = 0u;
    *p.loss_out =
        p.reduction == VPCE_SUM ? float(tot) : (c > 0 ? float(tot / double(c)) : __int_as_float(0x7fc00000));
  }
}

template <int G>
constexpr size_t fused_smem() {
  return size_t(kFusedWarps) * (kRingA + kRingB) * kFChunk + size_t(kFusedWarps) * (kRingA + kRingB) * 8 +
         size_t(kFusedWarps / G) * 2 * 8 + size_t(kFusedWarps / G) * 2 * G * sizeof(float2);
}

}  // namespace

// Rows are handled by groups of kFusedGroup warps.
constexpr int kFusedGroup = 8;

bool fused_supported(const ShardSet& sh, int t, int elem) {
  for (int i = 0; i < t; ++i) {
    const long long wb = (sh.start[i + 1] - sh.start[i]) * elem;
    if ((reinterpret_cast<uintptr_t>(sh.ptr[i]) & 15u) || (sh.ld_bytes[i] & 15) || (wb & 15)) return false;
  }
  return true;
}

cudaError_t set_fused_smem() {
  cudaError_t e = cudaFuncSetAttribute(fused_kernel<float, kFusedGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(fused_smem<kFusedGroup>()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fused_kernel<__nv_bfloat16, kFusedGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(fused_smem<kFusedGroup>()));
}

void launch_prep(const long long* targets, long long s, long long V, long long ignore_index, Header* hdr,
                 int reduction, float* loss_out, cudaStream_t st) {
  prep_kernel<<<1, kPrepThreads, 0, st>>>(targets, s, V, ignore_index, hdr, reduction, loss_out);
}

// The L2-reuse variant: any row length (rows stream through per-warp rings
// twice, the second time from L2).  Expects launch_prep before it.
void launch_l2fused(const ShardSet& sh, bool bf16, int t, long long s, long long V, const long long* targets,
                    long long ignore_index, int reduction, float grad, float* lse, float* rowl, float* row_loss,
                    float* loss_out, Header* hdr, int sms, cudaStream_t st) {
  FusedParams p;
  p.sh = sh;
  p.t = t;
  p.s = s;
  p.V = V;
  p.targets = targets;
  p.ignore_index = ignore_index;
  p.reduction = reduction;
  p.grad = grad;
  p.lse = lse;
  p.rowl = rowl;
  p.row_loss = row_loss;
  p.loss_out = loss_out;
  p.hdr = hdr;
  constexpr int NG = kFusedWarps / kFusedGroup;
  const long long want = (s + NG - 1) / NG;
  const int grid = int(want < sms ? want : sms);
  if (bf16)
    fused_kernel<__nv_bfloat16, kFusedGroup>
        <<<grid, kFusedWarps * 32, fused_smem<kFusedGroup>(), st>>>(p);
  else
    fused_kernel<float, kFusedGroup><<<grid, kFusedWarps * 32, fused_smem<kFusedGroup>(), st>>>(p);
}

}  // namespace vpce
