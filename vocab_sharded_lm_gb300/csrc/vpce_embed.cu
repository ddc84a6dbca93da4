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
// the (id, row) pairs of up to kEmbChunk rows are sorted (each CTA sorts 1024
// of them in shared memory, bitonic, then merge-path rounds double the sorted
// width), one CTA marks where each id's run starts, and one warp per
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
constexpr int kSortBlock = 1024;  // keys sorted by one CTA before the merge rounds

// One CTA per kSortBlock keys: this block's (id << 32 | row) keys (kNoKey for
// padding and for ids outside [0, V)), bitonic-sorted in shared memory.
__global__ void __launch_bounds__(kSortBlock / 2) embed_block_sort_kernel(const long long* ids, int n, int n_pow2,
                                                                          long long V, unsigned long long* out) {
  __shared__ unsigned long long key[kSortBlock];
  const int len = n_pow2 < kSortBlock ? n_pow2 : kSortBlock;
  const int base = blockIdx.x * len;
  for (int k = threadIdx.x; k < len; k += blockDim.x) {
    const int g = base + k;
    unsigned long long v = kNoKey;
    if (g < n) {
      const long long id = ids[g];
      if (id >= 0 && id < V) v = (static_cast<unsigned long long>(id) << 32) | unsigned(g);
    }
    key[k] = v;
  }
  __syncthreads();
  for (int size = 2; size <= len; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int k = threadIdx.x; k < len / 2; k += blockDim.x) {
        const int lo = 2 * k - (k & (stride - 1));  // first element of this compare pair
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x = key[lo], y = key[hi];
        if ((x > y) == up) {
          key[lo] = y;
          key[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int k = threadIdx.x; k < len; k += blockDim.x) out[base + k] = key[k];
}

// One merge round: pairs of sorted runs of `width` keys become runs of
// 2 * width.  Each key's place is its index in its own run plus the number of
// keys of the partner run before it (a binary search; keys of the first run
// go before equal keys of the second, so the padding keys stay in order).
__global__ void embed_merge_kernel(const unsigned long long* in, unsigned long long* out, int width, int total) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int pair = i / (2 * width), base = pair * 2 * width;
  const int j = i - base;
  const bool first = j < width;
  const int own = first ? j : j - width;
  const unsigned long long* other = in + base + (first ? width : 0);
  const unsigned long long v = in[i];
  int lo = 0, hi = width;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (first ? (other[mid] < v) : (other[mid] <= v)) lo = mid + 1;
    else hi = mid;
  }
  out[base + own + lo] = v;
}

struct EmbedRunsParams {
  const unsigned long long* keys;  // [n_pow2] sorted
  int n_pow2;
  int* seg;                        // [kEmbChunk + 1] start of each distinct id's run; seg[n_seg] = end
  int* n_seg;
  int* heavy;                      // [kEmbChunk / kHeavyRows] runs longer than kHeavyRows (any order)
  int* n_heavy;
};

// One CTA: the start of every run of equal ids in the sorted keys (ids outside
// [0, V) sorted last as kNoKey and are dropped), and the list of long runs.
__global__ void __launch_bounds__(kSortThreads) embed_runs_kernel(const EmbedRunsParams p) {
  __shared__ int warp_sum[kSortThreads / 32];
  __shared__ int nh;
  const int tid = threadIdx.x;
  const unsigned long long* key = p.keys;
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
  if (tid == 0) nh = 0;
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
  const int total = warp_sum[kSortThreads / 32 - 1];
  if (tid == kSortThreads - 1) {
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
  __syncthreads();  // seg[] (global) is complete and visible to the block
  // the long runs, listed for the CTA-per-chunk kernel (their order does not
  // matter: each run's sum is formed on its own)
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

// Work items are (short run, 512 columns) pairs, one warp each: four
// 128-column chunks at once (four float4 accumulators per lane), the run's
// rows in ascending order two at a time, so eight independent loads are in
// flight per lane; then one add into the id's row of the gradient table.
// The order of the additions per element does not depend on the grouping.
__global__ void __launch_bounds__(kEmbThreads) embed_accum_kernel(const __grid_constant__ EmbedAccParams p) {
  __shared__ long long start[VPCE_MAX_SHARDS + 1];
  for (int i = threadIdx.x; i <= p.t; i += kEmbThreads) start[i] = p.gsh.start[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  constexpr int kU = 4;  // 128-column chunks per task
  const long long nseg = *p.n_seg;
  const long long ngrp = (p.h + 128 * kU - 1) / (128 * kU);
  const long long tasks = nseg * ngrp;
  const long long nwarps = (long long)gridDim.x * (kEmbThreads / 32);
  for (long long q = (long long)blockIdx.x * (kEmbThreads / 32) + (threadIdx.x >> 5); q < tasks; q += nwarps) {
    const long long sgi = q / ngrp;
    const long long c0 = (q - sgi * ngrp) * (128 * kU) + 4 * lane;
    const int a = p.seg[sgi], b = p.seg[sgi + 1];
    if (b - a > kHeavyRows) continue;  // long runs: embed_heavy_kernel
    bool in[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) in[u] = c0 + 128 * u < p.h;
    float4 acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    int k = a;
    for (; k + 2 <= b; k += 2) {
      const int r0 = int(p.keys[k] & 0xffffffffu), r1 = int(p.keys[k + 1] & 0xffffffffu);
      float4 g0[kU], g1[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        g0[u] = in[u] ? grad4(p, r0, c0 + 128 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        g1[u] = in[u] ? grad4(p, r1, c0 + 128 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        acc[u].x += g0[u].x;
        acc[u].y += g0[u].y;
        acc[u].z += g0[u].z;
        acc[u].w += g0[u].w;
        acc[u].x += g1[u].x;
        acc[u].y += g1[u].y;
        acc[u].z += g1[u].z;
        acc[u].w += g1[u].w;
      }
    }
    if (k < b) {
      const int r0 = int(p.keys[k] & 0xffffffffu);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float4 g = in[u] ? grad4(p, r0, c0 + 128 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        acc[u].x += g.x;
        acc[u].y += g.y;
        acc[u].z += g.z;
        acc[u].w += g.w;
      }
    }
    const long long id = static_cast<long long>(p.keys[a] >> 32);
    const int i = shard_of(start, p.t, id);
    float* dst = reinterpret_cast<float*>(const_cast<unsigned char*>(p.gsh.ptr[i]) +
                                          (id - start[i]) * p.gsh.ld_bytes[i]) + c0;
    float4 o[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (in[u]) o[u] = *reinterpret_cast<const float4*>(dst + 128 * u);
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (in[u]) {
        o[u].x += acc[u].x;
        o[u].y += acc[u].y;
        o[u].z += acc[u].z;
        o[u].w += acc[u].w;
        *reinterpret_cast<float4*>(dst + 128 * u) = o[u];
      }
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
  return 2 * round256(sizeof(unsigned long long) * kEmbChunk) + round256(sizeof(int) * (kEmbChunk + 1)) +
         round256(sizeof(int) * (kEmbChunk / kHeavyRows)) + 256;
}

cudaError_t set_embed_smem() { return cudaSuccess; }

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
  const size_t kb = round256(sizeof(unsigned long long) * kEmbChunk);
  unsigned long long* keys_a = reinterpret_cast<unsigned long long*>(w);
  unsigned long long* keys_b = reinterpret_cast<unsigned long long*>(w + kb);
  int* seg = reinterpret_cast<int*>(w + 2 * kb);
  int* heavy = reinterpret_cast<int*>(w + 2 * kb + round256(sizeof(int) * (kEmbChunk + 1)));
  int* n_seg = reinterpret_cast<int*>(w + 2 * kb + round256(sizeof(int) * (kEmbChunk + 1)) +
                                      round256(sizeof(int) * (kEmbChunk / kHeavyRows)));
  int* n_heavy = n_seg + 1;
  const int eb = grad_bf16 ? 2 : 4;
  for (long long r0 = 0; r0 < s; r0 += kEmbChunk) {
    const int n = int(s - r0 < kEmbChunk ? s - r0 : kEmbChunk);
    int n2 = 2;
    while (n2 < n) n2 <<= 1;
    // sort: blocks of kSortBlock keys, then merge rounds (ping-pong buffers)
    const int blk = n2 < kSortBlock ? n2 : kSortBlock;
    embed_block_sort_kernel<<<n2 / blk, kSortBlock / 2, 0, st>>>(ids + r0, n, n2, V, keys_a);
    unsigned long long* cur = keys_a;
    unsigned long long* nxt = keys_b;
    for (int width = blk; width < n2; width <<= 1) {
      embed_merge_kernel<<<(n2 + 255) / 256, 256, 0, st>>>(cur, nxt, width, n2);
      unsigned long long* tmp = cur;
      cur = nxt;
      nxt = tmp;
    }
    unsigned long long* keys = cur;
    EmbedRunsParams rp;
    rp.keys = keys;
    rp.n_pow2 = n2;
    rp.seg = seg;
    rp.n_seg = n_seg;
    rp.heavy = heavy;
    rp.n_heavy = n_heavy;
    embed_runs_kernel<<<1, kSortThreads, 0, st>>>(rp);
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
    const long long want = ((long long)n * ((h + 511) / 512) + kEmbThreads / 32 - 1) / (kEmbThreads / 32);
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
