// Forward of the vocab-parallel cross-entropy.
//
// "Distributed Training III: Model Parallelism" (CMU 11-868 Lecture 16
// notes), §5.5 "Embedding and output layer", and "LLM Internals" §7.3.4: each
// vocabulary shard reduces, per row, its maximum, its sum of exponentials and
// (on the one shard that holds it) the target logit; those three scalars per
// token combine into logsumexp - target without gathering the rows.
//
// Kernel 1 (partial_stats) streams every (shard, row) segment through shared
// memory with the bulk-copy engine and keeps an online (max, sum-exp) in fp32.
// Kernel 2 (combine) folds the t partials of each row in ascending shard order
// (the on-device stand-in for the pages' max / sum / sum all-reduces), masks
// ignore_index, and reduces the batch in a fixed order in fp64.
#include "vpce_chunk.cuh"

namespace vpce {

namespace {

// Walks the bulk-copy chunks of a warp's units in order: units whose row is
// ignored or whose aligned body is empty have no chunks.
struct ChunkCursor {
  long long u_end;
  UnitPos pos;
  unsigned off;
  Unit g;
  bool ok;

  // the first unit with chunks at or after the current position
  template <int EB>
  __device__ __forceinline__ void seek(const StatsParams& p) {
    ok = false;
    for (; pos.u < u_end; pos.step(p.s)) {
      g = make_unit_at(p.sh, pos.shard, pos.row, EB);
      if (g.body == 0) continue;
      if (__ldg(p.targets + g.row) == p.ignore_index) continue;
      off = 0;
      ok = true;
      return;
    }
  }
  template <int EB>
  __device__ __forceinline__ void next(const StatsParams& p) {
    off += kChunk;
    if (off >= g.body) {
      pos.step(p.s);
      seek<EB>(p);
    }
  }
  __device__ __forceinline__ unsigned bytes() const { return min(unsigned(kChunk), g.body - off); }
  __device__ __forceinline__ const unsigned char* src() const { return g.addr + g.head + off; }
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32, 1) partial_stats_kernel(const __grid_constant__ StatsParams p) {
  constexpr int EB = Elem<T>::kBytes;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* ring = smem + size_t(warp) * kStages * kChunk;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + size_t(kWarps) * kStages * kChunk) + warp * kStages;

  const long long nw = (long long)gridDim.x * kWarps;
  const long long gw = (long long)blockIdx.x * kWarps + warp;
  const long long u0 = p.units * gw / nw;
  const long long u1 = p.units * (gw + 1) / nw;

  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kStages; ++k) mbar_init(&bar[k], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t pol = policy_evict_first();

  ChunkCursor prod;
  prod.u_end = u1;
  prod.pos.at(u0, p.s);
  prod.seek<EB>(p);
  unsigned issued = 0;
#pragma unroll 1
  for (int k = 0; k < kStages && prod.ok; ++k) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[k], prod.bytes());
      bulk_load(ring + k * kChunk, prod.src(), prod.bytes(), &bar[k], pol);
    }
    ++issued;
    prod.next<EB>(p);
  }

  unsigned kc = 0;
  bool alive = true;
  UnitPos cur;
  cur.at(u0, p.s);
#pragma unroll 1
  for (; cur.u < u1 && alive; cur.step(p.s)) {
    const Unit g = make_unit_at(p.sh, cur.shard, cur.row, EB);
    const long long y = __ldg(p.targets + g.row);
    if (y == p.ignore_index) continue;
    const long long lo = p.sh.start[g.shard], hi = p.sh.start[g.shard + 1];
    const bool has_t = (y >= lo) && (y < hi);
    float zt = 0.f;
    if (has_t && lane == 0) zt = Elem<T>::load(g.addr + (y - lo) * EB);

    // ragged head / tail elements outside the 16-byte aligned body
    float m = -INFINITY, sm = 0.f;
    {
      const int hn = int(g.head) / EB, tn = int(g.tail) / EB;
      float x = -INFINITY;
      if (lane < hn) x = Elem<T>::load(g.addr + lane * EB);
      else if (lane >= 16 && lane - 16 < tn) x = Elem<T>::load(g.addr + g.head + g.body + (lane - 16) * EB);
      if (x > -INFINITY) {
        m = x;
        sm = 1.f;
      }
    }

#pragma unroll 1
    for (unsigned off = 0; off < g.body; off += kChunk) {
      const unsigned n = min(unsigned(kChunk), g.body - off);
      const int slot = int(kc % kStages);
      if (!mbar_wait_warp(&bar[slot], (kc / kStages) & 1u)) {
        alive = false;
        break;
      }
      stats_chunk<kChunk / 512>(ring + slot * kChunk, n, lane, m, sm, T());
      __syncwarp();
      if (prod.ok) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar[slot], prod.bytes());
          bulk_load(ring + slot * kChunk, prod.src(), prod.bytes(), &bar[slot], pol);
        }
        ++issued;
        prod.next<EB>(p);
      }
      ++kc;
    }
    if (!alive) break;
    warp_merge_ms(m, sm);
    if (lane == 0) {
      p.part[(long long)g.shard * p.s + g.row] = make_float2(m, sm);
      if (has_t) p.tgt[g.row] = zt;
    }
  }

  if (!alive) {
    // A wait gave up: record it, then give the loads still in flight a bounded
    // chance to land before this warp's shared memory is released.
    if (lane == 0) atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
    for (unsigned k = kc; k < issued; ++k) {
      if (!mbar_wait_warp(&bar[k % kStages], (k / kStages) & 1u)) break;
    }
  }
}

// Fixed-order sum of a double and an int over a block of kCombineThreads.
__device__ __forceinline__ void block_sum(double& v, int& c, double* sv, int* sc) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v += __shfl_down_sync(kFull, v, o);
    c += __shfl_down_sync(kFull, c, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = v;
    sc[warp] = c;
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int nw = kCombineThreads / 32;
    v = lane < nw ? sv[lane] : 0.0;
    c = lane < nw ? sc[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v += __shfl_down_sync(kFull, v, o);
      c += __shfl_down_sync(kFull, c, o);
    }
  }
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
  __shared__ double sv[kCombineThreads / 32];
  __shared__ int sc[kCombineThreads / 32];
  __shared__ bool last;
  const long long r = (long long)blockIdx.x * kCombineThreads + threadIdx.x;
  double v = 0.0;
  int c = 0;
  // the partial statistics ran before this kernel (stream order); if one of
  // their waits gave up, the partials are incomplete and every row's loss is NaN
  const bool timed_out = (__ldcg(&p.hdr->error_flag) & VPCE_FLAG_WAIT_TIMEOUT) != 0;
  if (r < p.s) {
    const long long y = p.targets[r];
    float rl = 0.f, lse = 0.f;
    if (y == p.ignore_index) {
      rl = 0.f;
    } else if (y < 0 || y >= p.V) {
      rl = __int_as_float(0x7fc00000);
      lse = rl;
      atomicOr(&p.hdr->error_flag, VPCE_FLAG_BAD_TARGET);
      v = double(rl);
    } else {
      // global max first, then the sum-exps rescaled to it, shards ascending
      float M = -INFINITY;
      for (int i = 0; i < p.t; ++i) M = fmaxf(M, p.part[(long long)i * p.s + r].x);
      float S = 0.f;
      for (int i = 0; i < p.t; ++i) {
        const float2 q = p.part[(long long)i * p.s + r];
        S += q.y * expf(q.x - M);
      }
      lse = M + logf(S);
      rl = lse - p.tgt[r];
      if (timed_out) rl = lse = __int_as_float(0x7fc00000);
      v = double(rl);
      c = 1;
    }
    p.lse[r] = lse;
    if (p.row_loss) p.row_loss[r] = rl;
  }
  block_sum(v, c, sv, sc);
  if (threadIdx.x == 0) {
    if (gridDim.x == 1) {
      last = true;
    } else {
      p.bsum[blockIdx.x] = v;
      p.bcnt[blockIdx.x] = c;
      __threadfence();
      last = atomicAdd(&p.hdr->ticket, 1u) == gridDim.x - 1;
    }
  }
  __syncthreads();
  if (!last) return;
  if (gridDim.x > 1) {
    __threadfence();
    v = 0.0;
    c = 0;
    for (int b = threadIdx.x; b < (int)gridDim.x; b += kCombineThreads) {
      v += __ldcg(p.bsum + b);
      c += __ldcg(p.bcnt + b);
    }
    __syncthreads();
    block_sum(v, c, sv, sc);
  }
  if (threadIdx.x == 0) {
    p.hdr->n_valid = c;
    p.hdr->loss_sum = v;
    p.hdr->reduction = p.reduction;
    p.hdr->ticket = 0u;
    float loss;
    if (p.reduction != VPCE_MEAN) loss = float(v);  // sum ('none' reports the sum when asked)
    else loss = c > 0 ? float(v / double(c)) : __int_as_float(0x7fc00000);
    if (p.loss_out != nullptr) *p.loss_out = loss;
  }
}

// One process's shards folded into one (max, sum exp) pair per row, shards
// in ascending order with the combine's arithmetic: M = max_i m_i, then
// S = sum_i se_i exp(m_i - M).  The result is the pair the process's whole
// vocabulary slice would give as one shard, so a process exchanges one
// pair per row however many shards it holds.
__global__ void __launch_bounds__(kCombineThreads) fold_kernel(const float2* part, int t, long long s, float2* out) {
  const long long r = (long long)blockIdx.x * kCombineThreads + threadIdx.x;
  if (r >= s) return;
  float M = -INFINITY;
  for (int i = 0; i < t; ++i) M = fmaxf(M, part[(long long)i * s + r].x);
  float S = 0.f;
  for (int i = 0; i < t; ++i) {
    const float2 q = part[(long long)i * s + r];
    S += q.y * expf(q.x - M);
  }
  out[r] = make_float2(M, S);
}

}  // namespace

void launch_fold(const float2* part, int t, long long s, float2* out, cudaStream_t st) {
  fold_kernel<<<int((s + kCombineThreads - 1) / kCombineThreads), kCombineThreads, 0, st>>>(part, t, s, out);
}

template <typename T>
void launch_stats(const StatsParams& p, int grid, cudaStream_t st) {
  partial_stats_kernel<T><<<grid, kWarps * 32, kRingSmem, st>>>(p);
}
template void launch_stats<float>(const StatsParams&, int, cudaStream_t);
template void launch_stats<__nv_bfloat16>(const StatsParams&, int, cudaStream_t);

void launch_combine(const CombineParams& p, int blocks, cudaStream_t st) {
  combine_kernel<<<blocks, kCombineThreads, 0, st>>>(p);
}

cudaError_t set_stats_smem() {
  cudaError_t e = cudaFuncSetAttribute(partial_stats_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kRingSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(partial_stats_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(kRingSmem));
}

}  // namespace vpce
