// Forward of the vocab-parallel cross-entropy.
//
// "Distributed Training III: Model Parallelism" (CMU 11-868 Lecture 16
// notes), §5.5 "Embedding and output layer", and "LLM Internals" §7.3.4: each
// vocabulary shard reduces, per row, its maximum, its sum of exponentials and
// (on the one shard that holds it) the target logit; those three scalars per
// token combine into logsumexp - target without gathering the rows.
//
// Kernel 1 (partial_stats) streams every (shard, row) segment into registers,
// one warp per segment at a time, and keeps an online (max, sum-exp) in fp32.
// The combine -- the t partials of a row folded in ascending shard order, the
// on-device stand-in for the pages' max / sum / sum all-reduces, with
// ignore_index masked -- runs in the same kernel, in the warp that adds a
// row's last partial, and its last block sums the batch in a fixed order.
// Kernel 2 (combine_kernel) is the same combine as a kernel of its own, for
// partials that come from elsewhere (other processes, the LM-head GEMM); its
// batch sum is fp64 over fixed blocks.
#include "vpce_chunk.cuh"

namespace vpce {

namespace {

// The combine of row r by the warp that adds its last partial (see
// StatsParams): the same arithmetic as combine_kernel -- the maximum, then the
// sum-exps rescaled to it in ascending shard order -- with the partials read
// by the lanes at once and broadcast.
__device__ __forceinline__ void combine_row_if_last(const StatsParams& p, long long r, long long y, int lane) {
  int last = 0;
  if (lane == 0) {
    // release: this warp's partial (and target logit) before its arrival;
    // acquire: for the last to arrive, every other shard's partial of the row.
    // (A fence before and after a plain atomic measured 0.3358 against
    // 0.3336 ms per forward call at s = 8192.)
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.row_cnt + r) : "memory");
    last = old == p.t - 1;
  }
  if (!__shfl_sync(kFull, last, 0)) return;
  __syncwarp();  // the other lanes' loads below come after lane 0's acquire
  const float2 none = make_float2(-INFINITY, 0.f);
  const float2 q0 = lane < p.t ? __ldcg(p.part + (long long)lane * p.s + r) : none;
  const float2 q1 = lane + 32 < p.t ? __ldcg(p.part + (long long)(lane + 32) * p.s + r) : none;
  float M = fmaxf(q0.x, q1.x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float S = 0.f;
  for (int i = 0; i < p.t; ++i) {
    const float qx = __shfl_sync(kFull, i < 32 ? q0.x : q1.x, i & 31);
    const float qy = __shfl_sync(kFull, i < 32 ? q0.y : q1.y, i & 31);
    S += qy * expf(qx - M);
  }
  if (lane != 0) return;
  float lse, rl;
  if (y < 0 || y >= p.V) {
    lse = rl = __int_as_float(0x7fc00000);
    atomicOr(&p.hdr->error_flag, VPCE_FLAG_BAD_TARGET);
  } else {
    lse = M + logf(S);
    rl = lse - __ldcg(p.tgt + r);
    atomicAdd(&p.hdr->n_valid, 1);
  }
  p.lse[r] = lse;
  p.tgt[r] = rl;  // the target logit's slot now holds the row loss
  if (p.row_loss) p.row_loss[r] = rl;
}

// Kernel 1: one warp per (shard, row) unit at a time.  Each lane loads
// U 16-byte vectors per step straight into registers (streaming loads) and
// folds them into its (max, sum-exp); a shuffle merge gives the unit's
// partial.  Many warps per SM keep the loads in flight, and a unit's first
// vectors are loaded together with its target (a unit whose row turns out to
// be ignored drops them), so a unit starts with one memory round trip.
// Measured on GB300 (forward call: this kernel, the combine and the header
// clear): bf16 at s = 8192, V = 128256 0.336 ms against 0.347 ms for a
// bulk-copy ring of 2 x 12 KB per warp with 8 warps per SM, 2.42 against
// 2.55 ms at s = 32768; fp32 at s = 16384 1.398 against 1.403 ms.  More
// warps per SM (4 blocks of 8 vectors per lane) measured slower for bf16
// (0.341 ms), one block of 16 slower still (0.356 ms).
template <typename T, int U, int B>
__global__ void __launch_bounds__(kRegThreads, B) partial_stats_kernel(const __grid_constant__ StatsParams p) {
  constexpr int EB = Elem<T>::kBytes;
  const int lane = threadIdx.x & 31;
  // the backward that follows may start its ring set-up and first loads on
  // SMs this grid leaves; it waits for this grid before reading its results
  grid_launch_dependents();
  WarpUnits w;
#pragma unroll 1
  for (w.start(p.s); w.u < p.units; w.next(p.s)) {
    const Unit g = make_unit_at(p.sh, w.shard, w.row, EB);
    const uint4* v = reinterpret_cast<const uint4*>(g.addr + g.head);
    const int nv = int(g.body >> 4);
    const long long y = __ldg(p.targets + g.row);
    uint4 q[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int idx = lane + 32 * j;
      q[j] = idx < nv ? __ldcs(v + idx) : neg_inf_vec(T());
    }
    if (y == p.ignore_index) {
      // an ignored row: no partials; its shard-0 unit writes its zeros
      if (p.row_cnt != nullptr && g.shard == 0 && lane == 0) {
        p.lse[g.row] = 0.f;
        p.tgt[g.row] = 0.f;
        if (p.row_loss) p.row_loss[g.row] = 0.f;
      }
      continue;
    }
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
    for (int base = 0;;) {
      stats_vecs<U>(q, m, sm, T());
      base += 32 * U;
      if (base >= nv) break;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int idx = base + lane + 32 * j;
        q[j] = idx < nv ? __ldcs(v + idx) : neg_inf_vec(T());
      }
    }
    warp_merge_ms(m, sm);
    if (lane == 0) {
      p.part[(long long)g.shard * p.s + g.row] = make_float2(m, sm);
      if (has_t) p.tgt[g.row] = zt;
    }
    if (p.row_cnt != nullptr) combine_row_if_last(p, g.row, y, lane);
  }
  if (p.row_cnt == nullptr) return;

  // ---- batch loss: the last block sums the row losses in a fixed order
  __shared__ float2 sv[kRegThreads / 32];
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&p.hdr->ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const double tot = cta_fixed_sum<kRegThreads / 32>(p.tgt, p.s, sv);
  if (threadIdx.x == 0) {
    const int cnt = __ldcg(&p.hdr->n_valid);
    p.hdr->loss_sum = tot;
    p.hdr->reduction = p.reduction;
    p.hdr->ticket = 0u;
    if (p.loss_out != nullptr)
      *p.loss_out = p.reduction != VPCE_MEAN ? float(tot)
                                             : (cnt > 0 ? float(tot / double(cnt)) : __int_as_float(0x7fc00000));
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
void launch_stats(const StatsParams& p, int sms, cudaStream_t st) {
  using S = StatsShape<T>;
  const long long warps = kRegThreads / 32;
  const long long want = (p.units + warps - 1) / warps;  // one warp per unit at a time
  const long long cap = (long long)sms * S::kBlocksPerSm;
  const int grid = int(want < cap ? (want > 0 ? want : 1) : cap);
  partial_stats_kernel<T, S::kVecs, S::kBlocksPerSm><<<grid, kRegThreads, 0, st>>>(p);
}
template void launch_stats<float>(const StatsParams&, int, cudaStream_t);
template void launch_stats<__nv_bfloat16>(const StatsParams&, int, cudaStream_t);

void launch_combine(const CombineParams& p, int blocks, cudaStream_t st) {
  combine_kernel<<<blocks, kCombineThreads, 0, st>>>(p);
}

}  // namespace vpce
