// Device-side building blocks shared by the vocab-parallel cross-entropy
// kernels: workspace layout, shard geometry, and thin inline-PTX wrappers for
// the Blackwell bulk-copy engine (cp.async.bulk, 1-D TMA) and mbarriers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/vpce.h"

namespace vpce {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e), for exp(x) = 2^(x log2 e)
constexpr unsigned kFull = 0xffffffffu;
// A pipeline wait gives up after this many SM cycles (about a second at 2 GHz);
// the kernel then records VPCE_FLAG_WAIT_TIMEOUT and stops.
constexpr long long kWaitLimitCycles = 2000000000LL;

// ---------------------------------------------------------------------------
// workspace: [Header | part float2[t][s] | tgt float[s] | lse float[s] |
//             block sums double[nb] | block counts int[nb]]; every piece
// starts on a 256-byte boundary.
// ---------------------------------------------------------------------------
struct Header {
  int n_valid;          // rows whose target is not ignore_index (and in range)
  int error_flag;       // VPCE_FLAG_* bits
  unsigned ticket;      // combine: blocks that have published their sums
  int reduction;        // vpce_reduction of the forward
  double loss_sum;      // fp64 sum of valid-row losses
};
static_assert(sizeof(Header) <= 256, "header must fit its slot");

constexpr int kCombineThreads = 256;

__host__ __device__ inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t cnt, part, tgt, lse, bsum, bcnt, total;
  __host__ __device__ WsLayout(int t, long long s) {
    const long long nb = s > 0 ? (s + kCombineThreads - 1) / kCombineThreads : 1;
    cnt = 256;  // per-row shard arrivals, right after the header (one clear covers both)
    part = cnt + round256(sizeof(int) * size_t(s));
    tgt = part + round256(sizeof(float2) * size_t(t) * size_t(s));
    lse = tgt + round256(sizeof(float) * size_t(s));
    bsum = lse + round256(sizeof(float) * size_t(s));
    bcnt = bsum + round256(sizeof(double) * size_t(nb));
    total = bcnt + round256(sizeof(int) * size_t(nb));
  }
};

// ---------------------------------------------------------------------------
// shard geometry passed by value to every kernel
// ---------------------------------------------------------------------------
struct ShardSet {
  const unsigned char* ptr[VPCE_MAX_SHARDS];  // shard base addresses
  long long ld_bytes[VPCE_MAX_SHARDS];        // row stride in bytes
  long long start[VPCE_MAX_SHARDS + 1];       // vocabulary offsets
};

// One (shard, row) unit: the row segment [addr, addr + head + body + tail).
// `head` and `tail` are the bytes before the first and after the last 16-byte
// boundary inside the segment; `body` is the 16-byte aligned middle that the
// bulk-copy engine streams.
struct Unit {
  const unsigned char* addr;
  long long row;
  int shard;
  unsigned head, body, tail;
};

// The unit of (shard, row), with no division (streaming kernels walk units
// in order and carry (shard, row) along: UnitPos).
__device__ __forceinline__ Unit make_unit_at(const ShardSet& sh, int shard, long long row, int elem) {
  Unit g;
  g.shard = shard;
  g.row = row;
  g.addr = sh.ptr[g.shard] + g.row * sh.ld_bytes[g.shard];
  const unsigned len = unsigned(sh.start[g.shard + 1] - sh.start[g.shard]) * unsigned(elem);
  unsigned head = unsigned((16u - (unsigned(reinterpret_cast<uintptr_t>(g.addr)) & 15u)) & 15u);
  if (head > len) head = len;
  g.head = head;
  g.body = ((len - head) / 16u) * 16u;
  g.tail = len - head - g.body;
  return g;
}

// Position u = shard * s + row of a walk over units in order: one division
// when the walk starts, none per step.
struct UnitPos {
  long long u, row;
  int shard;
  __device__ __forceinline__ void at(long long u0, long long s) {
    u = u0;
    shard = int(u0 / s);
    row = u0 - (long long)shard * s;
  }
  __device__ __forceinline__ void step(long long s) {
    ++u;
    if (++row == s) {
      row = 0;
      ++shard;
    }
  }
};


// ---------------------------------------------------------------------------
// inline PTX: mbarrier + bulk async copies (sm_90+ forms, valid on sm_103a)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Warp-uniform bounded wait for the phase with the given parity.  Returns
// false (on every lane) when the limit passed first.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  for (;;) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(kFull, clock64() - t0 > kWaitLimitCycles)) return false;
  }
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// global -> shared bulk copy completing on `bar` (bytes: multiple of 16,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// shared -> global bulk copy tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
               "r"(smem_addr(src_smem)), "r"(bytes), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Single-thread bounded wait.
__device__ __forceinline__ bool mbar_wait_thread(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}
// ---------------------------------------------------------------------------
// thread-block clusters: another CTA's shared memory and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of `p` (this CTA's shared memory) in CTA `rank`
__device__ __forceinline__ uint32_t cluster_addr(const void* p, unsigned rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}

// arrive on the mbarrier at `bar` in CTA `rank` without a release: for an
// arrival that only reports that this thread's earlier loads are done (their
// values already used).  A release at cluster scope would make the thread
// wait for a fence.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(const uint64_t* bar, unsigned rank) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr(bar, rank))
               : "memory");
}

// Stores into another CTA's shared memory (dst, bar: shared::cluster
// addresses) that count their bytes on that CTA's mbarrier: the barrier's
// phase completes only once the data has landed, so the sender needs no
// release fence.
__device__ __forceinline__ void st_async_f2(uint32_t dst, float a, float b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(dst), "f"(a),
               "f"(b), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t dst, float a, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(dst), "f"(a), "r"(bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Warp-uniform bounded wait for a phase completed by arrivals from any CTA
// of the cluster (acquire at cluster scope); false once the limit passed.
__device__ __forceinline__ bool mbar_wait_warp_cluster(uint64_t* bar, uint32_t parity) {
  if (__all_sync(kFull, mbar_try_wait_cluster(bar, parity))) return true;
  const long long t0 = clock64();
  for (;;) {
    if (__all_sync(kFull, mbar_try_wait_cluster(bar, parity))) return true;
    if (__any_sync(kFull, clock64() - t0 > kWaitLimitCycles)) return false;
  }
}

__device__ __forceinline__ float2 ld_cluster_f2(const float2* p, unsigned rank) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(cluster_addr(p, rank))
               : "memory");
  return v;
}

__device__ __forceinline__ float ld_cluster_f(const float* p, unsigned rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}

// every thread of every CTA of the cluster (no time limit: callers reach it
// only after their own bounded waits)
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 2^x on the special-function unit (ftz; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// packed fp32 pairs (sm_100+): one instruction for two IEEE fp32 operations
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Pack two floats into a bf16x2 word, round to nearest even; `a` -> low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  static constexpr int kPerVec = 4;
  __device__ static float load(const unsigned char* p) { return *reinterpret_cast<const float*>(p); }
  __device__ static void store(unsigned char* p, float v) { *reinterpret_cast<float*>(p) = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;
  __device__ static float load(const unsigned char* p) {
    return __uint_as_float(uint32_t(*reinterpret_cast<const unsigned short*>(p)) << 16);
  }
  __device__ static void store(unsigned char* p, float v) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
  }
};

// Unpack one 16-byte vector into floats.
__device__ __forceinline__ void unpack(const uint4& v, float (&x)[4], float) {
  x[0] = __uint_as_float(v.x);
  x[1] = __uint_as_float(v.y);
  x[2] = __uint_as_float(v.z);
  x[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float (&x)[8], __nv_bfloat16) {
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}
__device__ __forceinline__ uint4 pack(const float (&d)[4], float) {
  return make_uint4(__float_as_uint(d[0]), __float_as_uint(d[1]), __float_as_uint(d[2]), __float_as_uint(d[3]));
}
__device__ __forceinline__ uint4 pack(const float (&d)[8], __nv_bfloat16) {
  return make_uint4(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]), pack_bf16x2(d[4], d[5]),
                    pack_bf16x2(d[6], d[7]));
}

// (m, s) pairs of a running max and a sum of exp(x - m): merge two.
__device__ __forceinline__ void merge_ms(float& m, float& s, float om, float os) {
  const float M = fmaxf(m, om);
  const float a = (m == M) ? s : s * ex2((m - M) * kLog2e);
  const float b = (om == M) ? os : os * ex2((om - M) * kLog2e);
  m = M;
  s = a + b;
}

__device__ __forceinline__ void warp_merge_ms(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(kFull, m, o);
    const float os = __shfl_xor_sync(kFull, s, o);
    merge_ms(m, s, om, os);
  }
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream serialization attribute may start while the kernel ahead of it in
// the stream still runs; grid_dependency_wait() blocks the calling thread
// until that kernel has completed and its writes are visible (at once when
// launched without the attribute), and grid_launch_dependents() in the
// kernel ahead lets the dependent start.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// A compensated fp32 sum: hi is the plain recursive sum and lo gathers the
// rounding error of every addition (Knuth's TwoSum), so hi + lo carries
// about twice fp32's precision.  A batch loss over thousands of rows summed
// by one CTA in fp64 spent microseconds in GB300's few fp64 units (8.6 us at
// s = 8192, 29 us at s = 32768); these adds run on the fp32 pipes.
struct FSum {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float t = hi + x;
    const float z = t - hi;
    lo += (hi - (t - z)) + (x - z);
    hi = t;
  }
  __device__ __forceinline__ void add(const FSum& o) {
    add(o.hi);
    lo += o.lo;
  }
  // hi + lo in fp64; a non-finite hi (an inf or NaN row loss) as it is, since
  // lo is then NaN
  __device__ __forceinline__ double value() const { return isfinite(hi) ? double(hi) + double(lo) : double(hi); }
};

// Sum of v[0 .. n) by one CTA of NW warps, in a fixed order (a given n and NW
// always give the same bits): warp w takes the 256-element blocks w, w + NW,
// ...; lane l adds elements 8l .. 8l + 7 of each, in order, to its FSum; a
// fixed shuffle tree adds the lanes and thread 0 the warps in order.  The
// loads of 4 blocks per warp are issued before any of them is added (one L2
// round trip per pass).  v must be 16-byte aligned; it is read through L2
// (__ldcg), so values other CTAs wrote before a fence are seen.  `sv` holds
// NW float2 in shared memory.  Every thread of the CTA must call it; thread
// 0 gets the sum.
template <int NW>
__device__ __forceinline__ double cta_fixed_sum(const float* v, long long n, float2* sv) {
  constexpr int kSumBlocks = 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  FSum acc;
  const long long nb = (n + 255) / 256;
  for (long long b0 = warp; b0 < nb; b0 += (long long)NW * kSumBlocks) {
    float x[kSumBlocks][8];
#pragma unroll
    for (int i = 0; i < kSumBlocks; ++i) {
      const long long r0 = (b0 + (long long)i * NW) * 256 + lane * 8;
      if (r0 + 8 <= n) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(v + r0));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(v + r0) + 1);
        x[i][0] = a.x, x[i][1] = a.y, x[i][2] = a.z, x[i][3] = a.w;
        x[i][4] = b.x, x[i][5] = b.y, x[i][6] = b.z, x[i][7] = b.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[i][j] = r0 + j < n ? __ldcg(v + r0 + j) : 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < kSumBlocks; ++i) {
      if (b0 + (long long)i * NW >= nb) break;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc.add(x[i][j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FSum q;
    q.hi = __shfl_down_sync(kFull, acc.hi, o);
    q.lo = __shfl_down_sync(kFull, acc.lo, o);
    acc.add(q);
  }
  if (lane == 0) sv[warp] = make_float2(acc.hi, acc.lo);
  __syncthreads();
  double tot = 0.0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NW; ++i) {
      FSum w;
      w.hi = sv[i].x;
      w.lo = sv[i].y;
      tot += w.value();
    }
  }
  return tot;
}

}  // namespace vpce
