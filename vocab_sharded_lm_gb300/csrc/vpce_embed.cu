// Vocabulary-parallel input embedding, forward and backward.
//
// "Distributed Training III: Model Parallelism" (CMU 11-868 Lecture 16 notes),
// §5.5, and "LLM Internals" §7.3.4: the table [V, h] is split by vocabulary
// into t shards; card i looks up only the ids in its range, writes zeros
// elsewhere, and an all-reduce sums the cards.  With every shard on one GPU
// the sum has exactly one non-zero term per row, so the forward is a gather
// of that term: each warp finds the shard that holds its row's id and copies
// the row (16-byte vectors, streaming loads); an id in no shard's range
// gives a zero row and raises a flag bit.
//
// The backward (not on the pages; the adjoint of the lookup) adds each
// output-gradient row into the table row of its id.  It is deterministic:
// a single CTA sorts the (id, row) pairs of up to kEmbChunk rows in shared
// memory (bitonic), marks where each id's run starts, and one warp per
// (distinct id, 128 columns) then sums the id's rows in ascending row order
// and adds the sum into the fp32 gradient table.  Longer batches run chunk after chunk on
// the stream, so the accumulation order is fixed.
#include "vpce_kernels.cuh"

namespace vpce {

namespace {

constexpr int kEmbThreads = 256;
constexpr int kSortThreads = 1024;
constexpr int kEmbChunk = 16384;  // rows sorted per backward chunk (128 KB of keys)
constexpr unsigned long long kNoKey = ~0ull;
constexpr int kHeavyRows = 64;  // ids with more rows are summed by a whole CTA

struct EmbedFwdParams {
  ShardSet sh;        // table shards [w_i, h] (ld_bytes = row stride)
  int t;
  long long V;
  long long h;        // columns
  int eb;             // element bytes (2 or 4)
  const long long* ids;
  long long s;
  unsigned char* out;
  long long ld_out_bytes;
  int* flag;          // may be null
};

// shard that holds id (-1: none)
__device__ __forceinline__ int shard_of(const long long* start, int t, long long id) {
  if (id < start[0] || id >= start[t]) return -1;
  int lo = 0, hi = t;  // start[lo] <= id < start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= id) lo = mid;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kEmbThreads) embed_forward_kernel(const __grid_constant__ EmbedFwdParams p) {
  __shared__ long long start[VPCE_MAX_SHARDS + 1];
  __shared__ const unsigned char* base[VPCE_MAX_SHARDS];
  __shared__ long long ldb[VPCE_MAX_SHARDS];
  for (int i = threadIdx.x; i <= p.t; i += kEmbThreads) {
    start[i] = p.sh.start[i];
    if (i < p.t) {
      base[i] = p.sh.ptr[i];
      ldb[i] = p.sh.ld_bytes[i];
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long row_bytes = p.h * p.eb;
  const long long nwarps = (long long)gridDim.x * (kEmbThreads / 32);
  for (long long r = (long long)blockIdx.x * (kEmbThreads / 32) + (threadIdx.x >> 5); r < p.s; r += nwarps) {
    const long long id = p.ids[r];
    const int i = shard_of(start, p.t, id);
    unsigned char* dst = p.out + r * p.ld_out_bytes;
    const unsigned char* src = i >= 0 ? base[i] + (id - start[i]) * ldb[i] : nullptr;
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | row_bytes) & 15) == 0;
    if (i < 0 && lane == 0 && p.flag != nullptr) atomicOr(p.flag, VPCE_FLAG_BAD_TARGET);
    if (vec) {
      const long long nv = row_bytes >> 4;
      uint4* d = reinterpret_cast<uint4*>(dst);
      const uint4* sp = reinterpret_cast<const uint4*>(src);
      long long v = lane;
      for (; v + 96 < nv; v += 128) {  // four independent 16-byte loads in flight per lane
        uint4 a, b, c, e;
        if (i >= 0) {
          a = ld_stream(sp + v);
          b = ld_stream(sp + v + 32);
          c = ld_stream(sp + v + 64);
          e = ld_stream(sp + v + 96);
        } else {
          a = b = c = e = make_uint4(0u, 0u, 0u, 0u);
        }
        d[v] = a;
        d[v + 32] = b;
        d[v + 64] = c;
        d[v + 96] = e;
      }
      for (; v < nv; v += 32) d[v] = i >= 0 ? ld_stream(sp + v) : make_uint4(0u, 0u, 0u, 0u);
    } else if (p.eb == 2) {
      unsigned short* d = reinterpret_cast<unsigned short*>(dst);
      const unsigned short* sp = reinterpret_cast<const unsigned short*>(src);
      for (long long c = lane; c < p.h; c += 32) d[c] = i >= 0 ? sp[c] : (unsigned short)0;
    } else {
      unsigned* d = reinterpret_cast<unsigned*>(dst);
      const unsigned* sp = reinterpret_cast<const unsigned*>(src);
      for (long long c = lane; c < p.h; c += 32) d[c] = i >= 0 ? sp[c] : 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
struct EmbedSortParams {
  const long long* ids;  // this chunk's ids
  int n;                 // rows in this chunk (<= kEmbChunk)
  int n_pow2;            // n rounded up to a power of two (>= 2)
  long long V;
  unsigned long long* keys;  // [kEmbChunk] sorted (id << 32 | row), kNoKey past the valid ones
  int* seg;                  // [kEmbChunk + 1] start of each distinct id's run; seg[n_seg] = end
  int* n_seg;
  int* heavy;                // [kEmbChunk / kHeavyRows] runs longer than kHeavyRows (any order)
  int* n_heavy;
};

// One CTA: bitonic sort of the chunk's (id, row) keys in shared memory, then
// the start of every run of equal ids (ids outside [0, V) sort last and are
// dropped).
__global__ void __launch_bounds__(kSortThreads) embed_sort_kernel(const EmbedSortParams p) {
  extern __shared__ unsigned long long key[];
  __shared__ int warp_sum[kSortThreads / 32];
  const int tid = threadIdx.x;
  for (int k = tid; k < p.n_pow2; k += kSortThreads) {
    unsigned long long v = kNoKey;
    if (k < p.n) {
      const long long id = p.ids[k];
      if (id >= 0 && id < p.V) v = (static_cast<unsigned long long>(id) << 32) | unsigned(k);
    }
    key[k] = v;
  }
  __syncthreads();
  for (int size = 2; size <= p.n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int k = tid; k < p.n_pow2 / 2; k += kSortThreads) {
        const int lo = 2 * k - (k & (stride - 1));  // first element of this compare pair
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long a = key[lo], b = key[hi];
        if ((a > b) == up) {
          key[lo] = b;
          key[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  // run heads: a valid key whose id differs from its predecessor's
  const int per = (p.n_pow2 + kSortThreads - 1) / kSortThreads;
  const int k0 = tid * per;
  int cnt = 0;
  for (int k = k0; k < k0 + per && k < p.n_pow2; ++k) {
    const unsigned long long v = key[k];
    if (v != kNoKey && (k == 0 || (key[k - 1] >> 32) != (v >> 32))) ++cnt;
  }
  // exclusive scan of the per-thread counts (thread order = key order)
  int incl = cnt;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += x;
    }
    warp_sum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int pos = incl - cnt + (warp > 0 ? warp_sum[warp - 1] : 0);
  for (int k = k0; k < k0 + per && k < p.n_pow2; ++k) {
    const unsigned long long v = key[k];
    if (v != kNoKey && (k == 0 || (key[k - 1] >> 32) != (v >> 32))) p.seg[pos++] = k;
  }
  for (int k = tid; k < p.n_pow2 && k < kEmbChunk; k += kSortThreads) p.keys[k] = key[k];
  if (tid == kSortThreads - 1) {
    const int total = warp_sum[kSortThreads / 32 - 1];
    *p.n_seg = total;
    // end of the last run: the number of valid keys, i.e. the first kNoKey
    // of the sorted array (binary search)
    int lo = 0, hi = p.n_pow2;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (key[mid] == kNoKey) hi = mid;
      else lo = mid + 1;
    }
    p.seg[total] = lo;
  }
  // the long runs, listed for the CTA-per-chunk kernel (their order does not
  // matter: each run's sum is formed on its own)
  __shared__ int nh;
  if (tid == 0) nh = 0;
  __syncthreads();  // seg[] (global) is complete and visible to the block
  const int total = warp_sum[kSortThreads / 32 - 1];
  for (int j = tid; j < total; j += kSortThreads)
    if (p.seg[j + 1] - p.seg[j] > kHeavyRows) p.heavy[atomicAdd(&nh, 1)] = j;
  __syncthreads();
  if (tid == 0) *p.n_heavy = nh;
}

struct EmbedAccParams {
  const unsigned long long* keys;
  const int* seg;
  const int* n_seg;
  const int* heavy;
  const int* n_heavy;
  const unsigned char* grad;  // this chunk's output-gradient rows
  long long ld_grad_bytes;
  int grad_bf16;
  long long h;
  ShardSet gsh;  // fp32 gradient table shards (ld_bytes = row stride)
  int t;
};

__device__ __forceinline__ float4 grad4(const EmbedAccParams& p, int row, long long c) {
  const unsigned char* base = p.grad + (long long)row * p.ld_grad_bytes;
  if (p.grad_bf16) {
    const uint2 w = *reinterpret_cast<const uint2*>(base + c * 2);
    return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
  }
  return *reinterpret_cast<const float4*>(base + c * 4);
}

// Work items are (distinct id, 128-column chunk) pairs, one warp each: the
// chunk's sum over the id's rows in ascending row order (eight rows loaded
// ahead, added in order), then one add into the id's row of the gradient
// table.  Splitting by columns spreads a frequent id over many warps; the
// order of the additions does not depend on the split.
__global__ void __launch_bounds__(kEmbThreads) embed_accum_kernel(const __grid_constant__ EmbedAccParams p) {
  __shared__ long long start[VPCE_MAX_SHARDS + 1];
  for (int i = threadIdx.x; i <= p.t; i += kEmbThreads) start[i] = p.gsh.start[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long nseg = *p.n_seg;
  const long long nch = (p.h + 127) / 128;
  const long long tasks = nseg * nch;
  const long long nwarps = (long long)gridDim.x * (kEmbThreads / 32);
  for (long long q = (long long)blockIdx.x * (kEmbThreads / 32) + (threadIdx.x >> 5); q < tasks; q += nwarps) {
    const long long sgi = q / nch;
    const long long c = (q - sgi * nch) * 128 + 4 * lane;
    const int a = p.seg[sgi], b = p.seg[sgi + 1];
    if (c >= p.h || b - a > kHeavyRows) continue;  // long runs: embed_heavy_kernel
    const long long id = static_cast<long long>(p.keys[a] >> 32);
    const int i = shard_of(start, p.t, id);
    float* dst = reinterpret_cast<float*>(const_cast<unsigned char*>(p.gsh.ptr[i]) +
                                          (id - start[i]) * p.gsh.ld_bytes[i]) + c;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int k = a;
    for (; k + 8 <= b; k += 8) {
      float4 g[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) g[u] = grad4(p, int(p.keys[k + u] & 0xffffffffu), c);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x += g[u].x;
        acc.y += g[u].y;
        acc.z += g[u].z;
        acc.w += g[u].w;
      }
    }
    for (; k < b; ++k) {
      const float4 g = grad4(p, int(p.keys[k] & 0xffffffffu), c);
      acc.x += g.x;
      acc.y += g.y;
      acc.z += g.z;
      acc.w += g.w;
    }
    float4 o = *reinterpret_cast<float4*>(dst);
    o.x += acc.x;
    o.y += acc.y;
    o.z += acc.z;
    o.w += acc.w;
    *reinterpret_cast<float4*>(dst) = o;
  }
}

// One CTA per (long run, 128-column chunk): warp w sums the w-th of eight
// contiguous slices of the run's rows (ascending), then warp 0 adds the eight
// partials in warp order and the result into the table row -- a fixed
// two-level order, so the sum does not depend on timing.
__global__ void __launch_bounds__(kEmbThreads) embed_heavy_kernel(const __grid_constant__ EmbedAccParams p) {
  __shared__ long long start[VPCE_MAX_SHARDS + 1];
  __shared__ float4 part[kEmbThreads / 32][32];
  for (int i = threadIdx.x; i <= p.t; i += kEmbThreads) start[i] = p.gsh.start[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kW = kEmbThreads / 32;
  const long long nch = (p.h + 127) / 128;
  const long long tasks = (long long)(*p.n_heavy) * nch;
  for (long long q = blockIdx.x; q < tasks; q += gridDim.x) {
    const long long hj = q / nch;
    const long long c = (q - hj * nch) * 128 + 4 * lane;
    const int sgi = p.heavy[hj];
    const int a = p.seg[sgi], b = p.seg[sgi + 1];
    const int n = b - a;
    const int lo = a + int((long long)n * warp / kW), hi = a + int((long long)n * (warp + 1) / kW);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < p.h) {
      int k = lo;
      for (; k + 8 <= hi; k += 8) {
        float4 g[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) g[u] = grad4(p, int(p.keys[k + u] & 0xffffffffu), c);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc.x += g[u].x;
          acc.y += g[u].y;
          acc.z += g[u].z;
          acc.w += g[u].w;
        }
      }
      for (; k < hi; ++k) {
        const float4 g = grad4(p, int(p.keys[k] & 0xffffffffu), c);
        acc.x += g.x;
        acc.y += g.y;
        acc.z += g.z;
        acc.w += g.w;
      }
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && c < p.h) {
      float4 tot = part[0][lane];
#pragma unroll
      for (int u = 1; u < kW; ++u) {
        tot.x += part[u][lane].x;
        tot.y += part[u][lane].y;
        tot.z += part[u][lane].z;
        tot.w += part[u][lane].w;
      }
      const long long id = static_cast<long long>(p.keys[a] >> 32);
      const int i = shard_of(start, p.t, id);
      float* dst = reinterpret_cast<float*>(const_cast<unsigned char*>(p.gsh.ptr[i]) +
                                            (id - start[i]) * p.gsh.ld_bytes[i]) + c;
      float4 o = *reinterpret_cast<float4*>(dst);
      o.x += tot.x;
      o.y += tot.y;
      o.z += tot.z;
      o.w += tot.w;
      *reinterpret_cast<float4*>(dst) = o;
    }
    __syncthreads();
  }
}

}  // namespace

size_t embed_bwd_workspace_bytes() {
  return round256(sizeof(unsigned long long) * kEmbChunk) + round256(sizeof(int) * (kEmbChunk + 1)) +
         round256(sizeof(int) * (kEmbChunk / kHeavyRows)) + 256;
}

cudaError_t set_embed_smem() {
  return cudaFuncSetAttribute(embed_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(sizeof(unsigned long long) * kEmbChunk));
}

void launch_embed_forward(const ShardSet& sh, int t, long long V, long long h, int eb, const long long* ids,
                          long long s, void* out, long long ld_out, int* flag, int sms, cudaStream_t st) {
  EmbedFwdParams p;
  p.sh = sh;
  p.t = t;
  p.V = V;
  p.h = h;
  p.eb = eb;
  p.ids = ids;
  p.s = s;
  p.out = static_cast<unsigned char*>(out);
  p.ld_out_bytes = ld_out * eb;
  p.flag = flag;
  const long long want = (s + kEmbThreads / 32 - 1) / (kEmbThreads / 32);
  const long long cap = (long long)sms * 8;
  embed_forward_kernel<<<int(want < cap ? want : cap), kEmbThreads, 0, st>>>(p);
}

// Chunk after chunk: sort, then accumulate.  Returns the last launch error.
cudaError_t launch_embed_backward(const void* grad, int grad_bf16, long long ld_grad, const long long* ids,
                                  long long s, const ShardSet& gsh, int t, long long V, long long h, void* ws,
                                  int sms, cudaStream_t st) {
  unsigned char* w = static_cast<unsigned char*>(ws);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(w);
  int* seg = reinterpret_cast<int*>(w + round256(sizeof(unsigned long long) * kEmbChunk));
  int* heavy = reinterpret_cast<int*>(w + round256(sizeof(unsigned long long) * kEmbChunk) +
                                      round256(sizeof(int) * (kEmbChunk + 1)));
  int* n_seg = reinterpret_cast<int*>(w + round256(sizeof(unsigned long long) * kEmbChunk) +
                                      round256(sizeof(int) * (kEmbChunk + 1)) +
                                      round256(sizeof(int) * (kEmbChunk / kHeavyRows)));
  int* n_heavy = n_seg + 1;
  const int eb = grad_bf16 ? 2 : 4;
  for (long long r0 = 0; r0 < s; r0 += kEmbChunk) {
    const int n = int(s - r0 < kEmbChunk ? s - r0 : kEmbChunk);
    int n2 = 2;
    while (n2 < n) n2 <<= 1;
    EmbedSortParams sp;
    sp.ids = ids + r0;
    sp.n = n;
    sp.n_pow2 = n2;
    sp.V = V;
    sp.keys = keys;
    sp.seg = seg;
    sp.n_seg = n_seg;
    sp.heavy = heavy;
    sp.n_heavy = n_heavy;
    embed_sort_kernel<<<1, kSortThreads, sizeof(unsigned long long) * n2, st>>>(sp);
    EmbedAccParams ap;
    ap.keys = keys;
    ap.seg = seg;
    ap.n_seg = n_seg;
    ap.heavy = heavy;
    ap.n_heavy = n_heavy;
    ap.grad = static_cast<const unsigned char*>(grad) + r0 * ld_grad * eb;
    ap.ld_grad_bytes = ld_grad * eb;
    ap.grad_bf16 = grad_bf16;
    ap.h = h;
    ap.gsh = gsh;
    ap.t = t;
    const long long want = ((long long)n * ((h + 127) / 128) + kEmbThreads / 32 - 1) / (kEmbThreads / 32);
    const long long cap = (long long)sms * 8;
    embed_accum_kernel<<<int(want < cap ? want : cap), kEmbThreads, 0, st>>>(ap);
    const long long hwant = (long long)(n / (kHeavyRows + 1) + 1) * ((h + 127) / 128);
    embed_heavy_kernel<<<int(hwant < cap ? hwant : cap), kEmbThreads, 0, st>>>(ap);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace vpce
