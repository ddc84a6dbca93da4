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
// width); one CTA marks where each id's run starts, lists the long runs and
// groups the short ones; one persistent kernel then sums every run in a fixed
// order and adds the sum into the fp32 gradient table, streaming the rows
// through shared memory with cp.async.  Longer batches run chunk after chunk
// on the stream, so the accumulation order is fixed.
#include "vpce_kernels.cuh"

namespace vpce {

namespace {

constexpr int kEmbThreads = 256;
constexpr int kSortThreads = 1024;
constexpr int kEmbChunk = 16384;  // rows sorted per backward chunk (128 KB of keys)
constexpr unsigned long long kNoKey = ~0ull;
constexpr int kHeavyRows = 64;  // ids with more rows are summed by a whole CTA
constexpr int kGroupRows = 16;  // short-run tasks: runs starting in this many consecutive sorted rows

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
  int* gstart;                     // [kEmbChunk / kGroupRows + 1] first run of each group of kGroupRows rows
  int* n_grp;
  unsigned* work;                  // [2] the accumulation's task counters, cleared here
  Header* hdr;                     // error flag (cleared when `first`)
  int first;                       // first chunk of the call
  ShardSet gsh;                    // fp32 gradient table shards
  int t;
  unsigned long long* rtab;        // [kEmbChunk] each run's gradient-table row (address)
};

// One CTA: the start of every run of equal ids in the sorted keys (ids outside
// [0, V) sorted last as kNoKey and are dropped), and the list of long runs.
__global__ void __launch_bounds__(kSortThreads) embed_runs_kernel(const __grid_constant__ EmbedRunsParams p) {
  __shared__ int warp_sum[kSortThreads / 32];
  __shared__ int nh;
  __shared__ long long start[VPCE_MAX_SHARDS + 1];
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
  for (int i = tid; i <= p.t; i += kSortThreads) start[i] = p.gsh.start[i];
  if (tid == 0) {
    nh = 0;
    p.work[0] = 0u;
    p.work[1] = 0u;
    if (p.first) p.hdr->error_flag = 0;
  }
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
  for (int j = tid; j < total; j += kSortThreads) {
    if (p.seg[j + 1] - p.seg[j] > kHeavyRows) p.heavy[atomicAdd(&nh, 1)] = j;
    // the run's row of the gradient table (every key here has an id in range)
    const long long id = static_cast<long long>(key[p.seg[j]] >> 32);
    const int i = shard_of(start, p.t, id);
    p.rtab[j] = reinterpret_cast<unsigned long long>(p.gsh.ptr[i] + (id - start[i]) * p.gsh.ld_bytes[i]);
  }
  // groups of kGroupRows sorted rows: group g holds the runs that start in
  // [g kGroupRows, (g + 1) kGroupRows); gstart[g] is its first run
  const int nvalid = p.seg[total];
  const int ngrp = (nvalid + kGroupRows - 1) / kGroupRows;
  for (int j = tid; j < total; j += kSortThreads) {
    const int g_lo = j == 0 ? 0 : p.seg[j - 1] / kGroupRows + 1, g_hi = p.seg[j] / kGroupRows;
    for (int g = g_lo; g <= g_hi; ++g) p.gstart[g] = j;
  }
  for (int g = (total > 0 ? p.seg[total - 1] / kGroupRows + 1 : 0) + tid; g <= ngrp; g += kSortThreads)
    p.gstart[g] = total;
  __syncthreads();
  if (tid == 0) {
    *p.n_heavy = nh;
    *p.n_grp = ngrp;
  }
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
  const int* gstart;
  const int* n_grp;
  const unsigned long long* rtab;  // each run's gradient-table row
  unsigned* work;                  // [2] task counters (zero at launch)
  Header* hdr;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, unsigned src_bytes) {
  // src_bytes < 16 zero-fills the rest of the 16 bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem)), "l"(gmem), "r"(src_bytes)
               : "memory");
}
// the mbarrier receives this thread's arrival once all its earlier cp.async
// copies have landed
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

constexpr int kAWarps = 8;
constexpr int kAThreads = kAWarps * 32;
constexpr int kShortCols = 256;  // columns per short-run task (8 per lane)
constexpr int kHeavyCols = 256;  // columns per long-run CTA task (8 per lane)
constexpr int kTRing = 8;        // runs (table slices) in flight per warp, at most 32

// A lane's share of a row slice of COLS columns, staged as 16-byte pieces:
// piece pc of lane l starts at column c0 + (32 pc + l) 16 / EB, so that a
// warp's piece pc is one contiguous span.  The lane's columns form COLS / 128
// quads of four (the fp32 table side): a bf16 piece holds quads 2 pc and
// 2 pc + 1, an fp32 piece is one quad.  Accumulator acc[4 q + e] is column e
// of quad q.
template <int EB, int COLS>
struct Slice {
  static constexpr int kPieces = COLS * EB / 512;
  static constexpr int kQuads = COLS / 128;
  static __device__ __forceinline__ long long piece_col(long long c0, int lane, int pc) {
    return c0 + (32LL * pc + lane) * (16 / EB);
  }
  static __device__ __forceinline__ long long quad_col(long long c0, int lane, int qd) {
    return EB == 2 ? c0 + 8 * lane + 4 * (qd & 1) + 256 * (qd >> 1) : c0 + 4 * lane + 128 * qd;
  }
};

template <int EB>
struct AccCfg {
  static constexpr int kRingBytes = EB == 2 ? 4096 : 8192;  // per warp, shared by both phases
  static constexpr int kRS = kRingBytes / (kShortCols * EB);  // short-run row slices in flight
  static constexpr int kRH = kRingBytes / (kHeavyCols * EB);  // long-run row slices in flight
};

template <int EB>
struct AccSmem {
  uint4 ring[kAWarps][AccCfg<EB>::kRingBytes / 16];  // slot-major: [slot][piece][lane]
  float4 table[kAWarps][kTRing][kShortCols / 128][32];
  float4 part[kAWarps][kHeavyCols / 128][32];
  uint64_t bar_s[kAWarps][AccCfg<EB>::kRS];
  uint64_t bar_h[kAWarps][AccCfg<EB>::kRH];
  unsigned task;
};

// A lane's view of 64 consecutive entries of an array, starting at a
// warp-uniform index that only moves forward: entries base + lane and
// base + 32 + lane, so that the next 32 are already on their way.
template <typename T>
struct Window {
  const T* a;
  long long n;  // entries [0, n) exist
  long long base;
  T cur, nxt;
  __device__ __forceinline__ T ld(long long i) const { return i < n ? a[i] : T(0); }
  __device__ __forceinline__ void init(const T* arr, long long len, long long k, int lane) {
    a = arr;
    n = len;
    base = k;
    cur = ld(k + lane);
    nxt = ld(k + 32 + lane);
  }
  __device__ __forceinline__ T at(long long k, int lane) {  // k >= base, warp-uniform
    if (k - base >= 64) {
      base = k;
      cur = ld(k + lane);
      nxt = ld(k + 32 + lane);
    } else if (k - base >= 32) {
      base += 32;
      cur = nxt;
      nxt = ld(base + 32 + lane);
    }
    return __shfl_sync(kFull, cur, int(k - base));
  }
  // entries k and k + 1, leaving the window at or before k
  __device__ __forceinline__ void pair(long long k, int lane, T& v0, T& v1) {
    const T a0 = at(k, lane);
    const int d = int(k - base);
    const T c1 = __shfl_sync(kFull, cur, (d + 1) & 31);
    const T n0 = __shfl_sync(kFull, nxt, 0);
    v0 = a0;
    v1 = d < 31 ? c1 : n0;
  }
};

// One lane's cp.async copies of one row slice into ring slot `slot`, and its
// arrival on the slot's mbarrier once they land.  Columns at or past h are
// zero-filled, nothing is read there.
template <int EB, int COLS>
__device__ __forceinline__ void stage_row(uint4* ring, int slot, int lane, const unsigned char* grow, long long c0,
                                          long long h, uint64_t* bar) {
  using S = Slice<EB, COLS>;
#pragma unroll
  for (int pc = 0; pc < S::kPieces; ++pc) {
    const long long col = S::piece_col(c0, lane, pc);
    const long long left = (h - col) * EB;
    const unsigned bytes = left >= 16 ? 16u : (left > 0 ? unsigned(left) : 0u);
    cp_async16(&ring[(slot * S::kPieces + pc) * 32 + lane], bytes ? grow + col * EB : grow, bytes);
  }
  cp_async_arrive(bar);
}

// acc += the lane's share of the row slice in ring slot `slot`
template <int EB, int COLS>
__device__ __forceinline__ void add_row(const uint4* ring, int slot, int lane, float* acc) {
  using S = Slice<EB, COLS>;
#pragma unroll
  for (int pc = 0; pc < S::kPieces; ++pc) {
    const uint4 v = ring[(slot * S::kPieces + pc) * 32 + lane];
    if (EB == 2) {
      float* a = acc + 8 * pc;
      a[0] += bf16_lo(v.x);
      a[1] += bf16_hi(v.x);
      a[2] += bf16_lo(v.y);
      a[3] += bf16_hi(v.y);
      a[4] += bf16_lo(v.z);
      a[5] += bf16_hi(v.z);
      a[6] += bf16_lo(v.w);
      a[7] += bf16_hi(v.w);
    } else {
      float* a = acc + 4 * pc;
      a[0] += __uint_as_float(v.x);
      a[1] += __uint_as_float(v.y);
      a[2] += __uint_as_float(v.z);
      a[3] += __uint_as_float(v.w);
    }
  }
}

// Every run's sum, added into its id's row of the fp32 gradient table, in
// one persistent launch.  Work is handed out through two counters.  First
// the long runs (more than kHeavyRows rows): one CTA per (run, kHeavyCols
// columns), each warp summing a contiguous eighth of the run and warp 0
// adding the eight partials in warp order.  Then the short runs: one warp
// per (group of the runs that start in kGroupRows consecutive sorted rows,
// kShortCols columns).  A warp streams its rows through a shared-memory
// ring: each lane copies its own 16-byte pieces with cp.async and the copy
// of the next row is issued as soon as a slot frees, across run boundaries;
// a run's table slice comes in with its first row, and the sum of the run's
// rows, in ascending order, is added to it after the run's last row.  Each
// element's sum has a fixed order whichever CTA or warp does the task.
template <int EB>
__global__ void __launch_bounds__(kAThreads) embed_accum_kernel(const __grid_constant__ EmbedAccParams p) {
  using C = AccCfg<EB>;
  using SS = Slice<EB, kShortCols>;
  using SH = Slice<EB, kHeavyCols>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AccSmem<EB>& sm = *reinterpret_cast<AccSmem<EB>*>(smem_raw);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint4* ring = sm.ring[w];
  if (lane == 0) {
    for (int k = 0; k < C::kRS; ++k) mbar_init(&sm.bar_s[w][k], 32);
    for (int k = 0; k < C::kRH; ++k) mbar_init(&sm.bar_h[w][k], 32);
    fence_mbar_init();
  }
  __syncthreads();
  const long long h = p.h;
  const int total = *p.n_seg;
  const long long nkeys = p.seg[total];  // valid keys
  bool ok = true;

  // ---- long runs: CTA tasks
  {
    const long long ncb = (h + kHeavyCols - 1) / kHeavyCols;
    const long long n_ht = (long long)(*p.n_heavy) * ncb;
    unsigned issued = 0, consumed = 0;
    for (;;) {
      if (threadIdx.x == 0) sm.task = atomicAdd(&p.work[0], 1u);
      __syncthreads();
      const long long q = sm.task;
      __syncthreads();
      if (q >= n_ht) break;
      const long long hj = q / ncb;
      const long long c0 = (q - hj * ncb) * kHeavyCols;
      const int sgi = p.heavy[hj];
      const int ra = p.seg[sgi], n = p.seg[sgi + 1] - ra;
      const int lo = ra + int((long long)n * w / kAWarps), hi = ra + int((long long)n * (w + 1) / kAWarps);
      float* trow = nullptr;
      float4 tq[SH::kQuads];
#pragma unroll
      for (int qd = 0; qd < SH::kQuads; ++qd) tq[qd] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (w == 0) {
        trow = reinterpret_cast<float*>(p.rtab[sgi]);
#pragma unroll
        for (int qd = 0; qd < SH::kQuads; ++qd) {
          const long long col = SH::quad_col(c0, lane, qd);
          if (col < h) tq[qd] = *reinterpret_cast<const float4*>(trow + col);
        }
      }
      float acc[4 * SH::kQuads];
#pragma unroll
      for (int e = 0; e < 4 * SH::kQuads; ++e) acc[e] = 0.f;
      Window<unsigned long long> kw;
      kw.init(p.keys, nkeys, lo, lane);
      long long pk = lo;
      for (int k = lo; k < hi && ok; ++k) {
        while (pk < hi && issued - consumed < unsigned(C::kRH)) {
          const unsigned long long key = kw.at(pk++, lane);
          const int slot = int(issued % C::kRH);
          stage_row<EB, kHeavyCols>(ring, slot, lane, p.grad + (long long)(key & 0xffffffffu) * p.ld_grad_bytes, c0, h,
                                    &sm.bar_h[w][slot]);
          ++issued;
        }
        const int slot = int(consumed % C::kRH);
        ok = mbar_wait_warp(&sm.bar_h[w][slot], (consumed / C::kRH) & 1u);
        if (ok) add_row<EB, kHeavyCols>(ring, slot, lane, acc);
        ++consumed;
      }
#pragma unroll
      for (int qd = 0; qd < SH::kQuads; ++qd)
        sm.part[w][qd][lane] = make_float4(acc[4 * qd], acc[4 * qd + 1], acc[4 * qd + 2], acc[4 * qd + 3]);
      __syncthreads();
      if (w == 0) {
#pragma unroll
        for (int qd = 0; qd < SH::kQuads; ++qd) {
          const long long col = SH::quad_col(c0, lane, qd);
          if (col >= h) continue;
          float4 tot = sm.part[0][qd][lane];
#pragma unroll
          for (int ww = 1; ww < kAWarps; ++ww) {
            const float4 v = sm.part[ww][qd][lane];
            tot.x += v.x;
            tot.y += v.y;
            tot.z += v.z;
            tot.w += v.w;
          }
          tq[qd].x += tot.x;
          tq[qd].y += tot.y;
          tq[qd].z += tot.z;
          tq[qd].w += tot.w;
          *reinterpret_cast<float4*>(trow + col) = tq[qd];
        }
      }
      __syncthreads();
    }
  }

  // ---- short runs: warp tasks
  const long long ncb = (h + kShortCols - 1) / kShortCols;
  const long long n_st = (long long)(*p.n_grp) * ncb;
  unsigned issued = 0, consumed = 0, run_ord = 0, flushed = 0;
  int r_len = 0;                 // run ordinal = lane (mod 32): its length ...
  unsigned long long r_dst = 0;  // ... and its table row
  float acc[4 * SS::kQuads];
  while (ok) {
    unsigned q = 0;
    if (lane == 0) q = atomicAdd(&p.work[1], 1u);
    q = __shfl_sync(kFull, q, 0);
    if (q >= n_st) break;
    const long long gi = q / ncb;
    const long long c0 = ((long long)q - gi * ncb) * kShortCols;
    const long long s1 = p.gstart[gi + 1];
    long long ps = p.gstart[gi];
    Window<int> sw;
    sw.init(p.seg, total + 1, ps, lane);
    Window<unsigned long long> pw;
    pw.init(p.rtab, total, ps, lane);
    Window<unsigned long long> kw;
    kw.init(p.keys, nkeys, sw.at(ps, lane), lane);
    long long pk = 0, pend = 0;
    bool pdone = false;
    // keeps the ring full: the rows of the task's short runs in order, a
    // run's table slice issued with its first row
    auto top_up = [&]() {
      while (!pdone && issued - consumed < unsigned(C::kRS)) {
        if (pk == pend) {
          int a = 0, b = 0;
          for (;;) {
            if (ps >= s1) {
              pdone = true;
              break;
            }
            sw.pair(ps, lane, a, b);
            if (b - a <= kHeavyRows) break;
            ++ps;  // a long run: its CTA tasks sum it
          }
          if (pdone || run_ord - flushed >= unsigned(kTRing)) break;
          const unsigned long long tp = pw.at(ps, lane);
          const float* trow = reinterpret_cast<const float*>(tp);
          const int ts = int(run_ord % kTRing);
#pragma unroll
          for (int qd = 0; qd < SS::kQuads; ++qd) {
            const long long col = SS::quad_col(c0, lane, qd);
            cp_async16(&sm.table[w][ts][qd][lane], col < h ? trow + col : trow, col < h ? 16u : 0u);
          }
          if (lane == int(run_ord & 31u)) {
            r_len = b - a;
            r_dst = tp;
          }
          ++run_ord;
          ++ps;
          pk = a;
          pend = b;
        }
        const unsigned long long key = kw.at(pk, lane);
        const int slot = int(issued % C::kRS);
        stage_row<EB, kShortCols>(ring, slot, lane, p.grad + (long long)(key & 0xffffffffu) * p.ld_grad_bytes, c0, h,
                                  &sm.bar_s[w][slot]);
        ++issued;
        ++pk;
      }
    };
    top_up();
    while (ok && consumed < issued) {
      const int ts = int(flushed % kTRing);
      const int len = __shfl_sync(kFull, r_len, int(flushed & 31u));
      float* trow = reinterpret_cast<float*>(__shfl_sync(kFull, r_dst, int(flushed & 31u)));
#pragma unroll
      for (int e = 0; e < 4 * SS::kQuads; ++e) acc[e] = 0.f;
      for (int r = 0; r < len; ++r) {
        const int slot = int(consumed % C::kRS);
        ok = mbar_wait_warp(&sm.bar_s[w][slot], (consumed / C::kRS) & 1u);
        if (!ok) break;
        add_row<EB, kShortCols>(ring, slot, lane, acc);
        ++consumed;
        top_up();
      }
      if (!ok) break;
      // the table slice arrived with the run's first row
#pragma unroll
      for (int qd = 0; qd < SS::kQuads; ++qd) {
        const long long col = SS::quad_col(c0, lane, qd);
        if (col >= h) continue;
        float4 o = sm.table[w][ts][qd][lane];
        o.x += acc[4 * qd + 0];
        o.y += acc[4 * qd + 1];
        o.z += acc[4 * qd + 2];
        o.w += acc[4 * qd + 3];
        *reinterpret_cast<float4*>(trow + col) = o;
      }
      ++flushed;
      top_up();
    }
  }
  if (!ok && lane == 0) atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
  cp_async_wait_all();  // nothing lands in shared memory after the CTA ends
}

int g_accum_ctas[2] = {1, 1};  // resident CTAs per SM of embed_accum_kernel<2>, <4>

}  // namespace

// Workspace: a header (its error flag is where vpce_read_error_flag looks),
// the two key buffers of the sort, the run starts, the long-run list, the
// group starts and the counters.
struct EmbedWs {
  Header* hdr;
  unsigned long long* keys_a;
  unsigned long long* keys_b;
  int* seg;
  int* heavy;
  int* gstart;
  unsigned long long* rtab;
  int* counts;  // n_seg, n_heavy, n_grp, work[2]
};

size_t embed_bwd_workspace_bytes() {
  return 256 + 2 * round256(sizeof(unsigned long long) * kEmbChunk) + round256(sizeof(int) * (kEmbChunk + 1)) +
         round256(sizeof(int) * (kEmbChunk / kHeavyRows)) + round256(sizeof(int) * (kEmbChunk / kGroupRows + 1)) +
         round256(sizeof(unsigned long long) * kEmbChunk) + 256;
}

EmbedWs embed_ws(void* ws) {
  unsigned char* w = static_cast<unsigned char*>(ws);
  EmbedWs e;
  e.hdr = reinterpret_cast<Header*>(w);
  w += 256;
  e.keys_a = reinterpret_cast<unsigned long long*>(w);
  w += round256(sizeof(unsigned long long) * kEmbChunk);
  e.keys_b = reinterpret_cast<unsigned long long*>(w);
  w += round256(sizeof(unsigned long long) * kEmbChunk);
  e.seg = reinterpret_cast<int*>(w);
  w += round256(sizeof(int) * (kEmbChunk + 1));
  e.heavy = reinterpret_cast<int*>(w);
  w += round256(sizeof(int) * (kEmbChunk / kHeavyRows));
  e.gstart = reinterpret_cast<int*>(w);
  w += round256(sizeof(int) * (kEmbChunk / kGroupRows + 1));
  e.rtab = reinterpret_cast<unsigned long long*>(w);
  w += round256(sizeof(unsigned long long) * kEmbChunk);
  e.counts = reinterpret_cast<int*>(w);
  return e;
}

cudaError_t set_embed_smem() {
  cudaError_t e = cudaFuncSetAttribute(embed_accum_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(sizeof(AccSmem<2>)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(embed_accum_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(sizeof(AccSmem<4>)));
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_accum_ctas[0], embed_accum_kernel<2>, kAThreads,
                                                      sizeof(AccSmem<2>));
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_accum_ctas[1], embed_accum_kernel<4>, kAThreads,
                                                      sizeof(AccSmem<4>));
  for (int& c : g_accum_ctas) c = c < 1 ? 1 : c;
  return e;
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
  const EmbedWs W = embed_ws(ws);
  int* n_seg = W.counts;
  int* n_heavy = W.counts + 1;
  int* n_grp = W.counts + 2;
  unsigned* work = reinterpret_cast<unsigned*>(W.counts + 3);
  const int eb = grad_bf16 ? 2 : 4;
  for (long long r0 = 0; r0 < s; r0 += kEmbChunk) {
    const int n = int(s - r0 < kEmbChunk ? s - r0 : kEmbChunk);
    int n2 = 2;
    while (n2 < n) n2 <<= 1;
    // sort: blocks of kSortBlock keys, then merge rounds (ping-pong buffers)
    const int blk = n2 < kSortBlock ? n2 : kSortBlock;
    embed_block_sort_kernel<<<n2 / blk, kSortBlock / 2, 0, st>>>(ids + r0, n, n2, V, W.keys_a);
    unsigned long long* cur = W.keys_a;
    unsigned long long* nxt = W.keys_b;
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
    rp.seg = W.seg;
    rp.n_seg = n_seg;
    rp.heavy = W.heavy;
    rp.n_heavy = n_heavy;
    rp.gstart = W.gstart;
    rp.n_grp = n_grp;
    rp.work = work;
    rp.hdr = W.hdr;
    rp.first = r0 == 0;
    rp.gsh = gsh;
    rp.t = t;
    rp.rtab = W.rtab;
    embed_runs_kernel<<<1, kSortThreads, 0, st>>>(rp);
    EmbedAccParams ap;
    ap.keys = keys;
    ap.seg = W.seg;
    ap.n_seg = n_seg;
    ap.heavy = W.heavy;
    ap.n_heavy = n_heavy;
    ap.grad = static_cast<const unsigned char*>(grad) + r0 * ld_grad * eb;
    ap.ld_grad_bytes = ld_grad * eb;
    ap.grad_bf16 = grad_bf16;
    ap.h = h;
    ap.gsh = gsh;
    ap.t = t;
    ap.gstart = W.gstart;
    ap.n_grp = n_grp;
    ap.rtab = W.rtab;
    ap.work = work;
    ap.hdr = W.hdr;
    // persistent: as many CTAs as fit take tasks until both lists are done
    if (grad_bf16)
      embed_accum_kernel<2><<<sms * g_accum_ctas[0], kAThreads, sizeof(AccSmem<2>), st>>>(ap);
    else
      embed_accum_kernel<4><<<sms * g_accum_ctas[1], kAThreads, sizeof(AccSmem<4>), st>>>(ap);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace vpce
